"""GB300 (sm_103a) implementation of R-KV's decode-time KV-cache compression
step: a C-ABI CUDA library (``librkv.so``, include/rkv.h) and its thin Python
binding (``rkv``).  Synthetic workloads live in ``workloads``."""
from .rkv import (RkvError, alloc_workspace, load, rkv_compress, rkv_compress_noalloc, rkv_gather,  # noqa: F401
                  rkv_get_device_status, rkv_score, rkv_select, rkv_timing_enable,
                  rkv_timing_read, rkv_workspace_init, rkv_workspace_size)
