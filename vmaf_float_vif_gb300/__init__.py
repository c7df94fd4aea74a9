"""vmaf_float_vif_gb300 -- the 4-scale float VIF score on one GB300 GPU.

The product is the C-ABI library ``libfvif.so`` (``include/fvif.h``) whose hot
path is hand-written sm_103a CUDA.  This package is its thin ctypes binding:
the functions below carry the C names and only marshal arguments; every step
of the score runs in the library's kernels.  There is no CPU path: when the
library is missing or cannot be loaded, every call raises.

PyTorch is used only as a source of device memory and streams (tensors'
``data_ptr()`` and ``torch.cuda.current_stream().cuda_stream``); numpy arrays
serve as host buffers.
"""
from ._lib import (  # noqa: F401
    FVIF_EINVAL, FVIF_ENOMEM, FVIF_ECUDA, FVIF_ETOOBIG, FVIF_OK, FvifError,
    NOALLOC_SCRATCH_BYTES, build, lib, fvif_score_noalloc,
    fvif_chunk_frames, fvif_create, fvif_debug_frame, fvif_destroy,
    fvif_get_taps, fvif_last_error, fvif_score, fvif_score_async,
    fvif_score_host, fvif_set_stream, fvif_strerror, fvif_profile_enable,
    fvif_profile_read, fvif_profile_host, HOST_PROFILE_COLUMNS,
    fvif_alu_probe, HostBuffer,
    fvif_debug_terms, fvif_create_ex, fvif_score_debug,
    fvif_default_options, FvifOptions, KERNEL_KINDS, Context, plane_sizes,
    fssim_auto_scale, fssim_decimated_size, fssim_decimate)
