"""Absorbed Multi-head Latent Attention decode for GB300 (sm_103a).

The compute lives in libmla.so (CUDA kernels behind the C ABI of
include/mla.h); this package is its ctypes binding with the same function
names.  Importing it fails loudly when the library has not been built
(see ``mla_absorbed_latent_gb300.build.build_library``).
"""

from ._binding import (  # noqa: F401
    D_C, D_NOPE, D_R, D_V, FMT, LIB_PATH, PAGE, MLA_NOALLOC_SCRATCH_BYTES,
    MLA_ERR_BOUNDS, MLA_ERR_CUDA, MLA_ERR_INVALID, MLA_ERR_TIMEOUT, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE,
    MLA_OK, MLA_KERNEL_CUDA_CORES, MLA_KERNEL_MMA, MLA_KERNEL_TCGEN05,
    MLAError, cache_struct, mla_absorb_weights, mla_cache_append, mla_cache_page_bytes, mla_cache_t, mla_decode,
    mla_cache_project_append, mla_cache_project_workspace_bytes,
    mla_decode_absorb_q, mla_decode_noalloc, mla_decode_plan, mla_decode_plan_workers, mla_decode_max_workers, mla_decode_q, mla_decode_q_workspace_bytes, mla_prefill, mla_prefill_workspace_bytes, mla_output_projection, mla_output_projection_workspace_bytes, mla_decode_attend, mla_decode_combine, mla_decode_kernel_kind, mla_decode_select_kernel,
    mla_decode_workspace_bytes,
    mla_get_device_status, mla_status_string, mla_wait_selftest, raw_library,
)
