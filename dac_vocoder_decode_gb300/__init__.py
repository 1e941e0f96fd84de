"""GB300-native DAC-style vocoder decoder: C-ABI CUDA library (libvocoder.so) + ctypes binding.

The CUDA library is the product; ``binding`` marshals arguments to it and
``workloads`` draws the seeded synthetic inputs."""
from .binding import (Vocoder, VocoderError, fold_params, load_library, vocoder_abi_version,  # noqa: F401
                      vocoder_create, vocoder_decode, vocoder_decode_host, vocoder_destroy,
                      vocoder_fold_weight_norm, vocoder_hop, vocoder_last_error,
                      vocoder_launches_per_decode, vocoder_op_conv1d, vocoder_op_conv_transpose1d,
                      vocoder_param_count, vocoder_param_shape, vocoder_profile,
                      vocoder_stitch, vocoder_stitched_length, vocoder_workspace_bytes,
                      vocoder_workspace_bytes_host)
