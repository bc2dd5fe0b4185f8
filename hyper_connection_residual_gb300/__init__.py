"""GB300 (sm_103a) hyper-connection read.

The read runs only in the CUDA library ``libhcread.so`` (hand-written kernels
behind the C ABI of ``include/hc_read.h``), and so does the Q2_0
matrix-vector product of ``include/hc_q2.h``.  This package is a thin ctypes
binding with the same entry-point names; it has no CPU path.
"""

from ._binding import (  # noqa: F401
    EXPORTS,
    HC_ERR_ALIGN,
    HC_ERR_ARG,
    HC_ERR_CUDA,
    HC_ERR_SHAPE,
    HC_ERR_TIMEOUT,
    HC_ERR_TOO_LARGE,
    HC_NOALLOC_MAX_T,
    HC_OK,
    HcError,
    Read,
    hc_graph_begin,
    hc_graph_destroy,
    hc_graph_end,
    hc_graph_launch,
    hc_q2_0_desc,
    hc_q2_0_matvec,
    hc_q2_0_matvec_batch,
    hc_q2_0_matvec_batch_plan,
    hc_read,
    hc_read_batch,
    hc_read_batch_groups,
    hc_read_batch_persistent,
    hc_read_batch_plan,
    hc_read_batch_q8,
    hc_read_batch_q8_groups,
    hc_read_batch_q8_plan,
    hc_read_q8,
    hc_read_q8_desc,
    hc_read_check,
    hc_read_create,
    hc_read_desc,
    hc_read_destroy,
    hc_read_error_word,
    hc_read_ex,
    hc_read_noalloc,
    hc_read_noalloc_check,
    hc_read_set_overlap,
    hc_read_down_tiles_bytes,
    hc_read_register_down_tiles,
    hc_read_forget_down_tiles,
    hc_read_up_tiles_bytes,
    hc_read_register_up_tiles,
    hc_read_forget_up_tiles,
    hc_read_set_wait_limit,
    hc_read_reset,
    hc_read_scratch_bytes,
    library_path,
    load,
    status_str,
)

GEOMETRIES = {"d2560_K320": (4, 2560, 320), "d4096_K512": (4, 4096, 512)}
