"""dense_fp16_tensor_gb300 -- fp16 TN GEMM for one GB300 (sm_103a).

    D(m,n) = C(m,n) + sum_k A(m,k) B(n,k)

A C-ABI library (include/gemm_tn.h, csrc/) with a ctypes binding of the same
names (``binding``) and a torch-tensor front end (``gemm`` for the in-place
form, ``gemm_scaled`` for D = alpha A.B^T + beta C, 2-D or batched 3-D, and
``gemm_host`` for the scaled form on CPU tensors, copies overlapped with the
GEMMs inside the library).  Build with
``build()``; there is no CPU or library fallback.
"""
from ._build import build  # noqa: F401
from .binding import (ACC_F16, ACC_F32, MAJOR_K, MAJOR_MN, PATH_AUTO, PATH_LARGE,  # noqa: F401
                      PATH_SKINNY, GemmTnError, gemm_tn, gemm_tn_check_device_error,
                      gemm_tn_ex, gemm_tn_last_kernels, gemm_tn_last_launch_count, gemm_tn_plan_path,
                      gemm_tn_status_string, gemm_tn_strided, gemm_tn_strided_ex, library_path,
                      make_options, gemm_tn_scaled, gemm_tn_batched, gemm_tn_batched_ex,
                      gemm_tn_host)


def gemm(*args, **kwargs):
    from .tensor_api import gemm as _gemm
    return _gemm(*args, **kwargs)


def gemm_scaled(*args, **kwargs):
    from .tensor_api import gemm_scaled as _gemm_scaled
    return _gemm_scaled(*args, **kwargs)


def gemm_host(*args, **kwargs):
    from .tensor_api import gemm_host as _gemm_host
    return _gemm_host(*args, **kwargs)
