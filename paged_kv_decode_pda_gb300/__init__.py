"""fp8 paged decode attention for NVIDIA GB300 (sm_103a).

Single-query attention over a paged fp8-e4m3 KV cache (16-token-multiple
blocks, per-sequence block tables, GQA up to 8) as a C-ABI library
(``include/pda.h``, ``libpda.so``) with hand-written sm_103a kernels: a
split-KV decode kernel, a log-sum-exp merge kernel and a host split-count
heuristic. This package is a thin ctypes binding; it performs no compute.
"""

from ._binding import (  # noqa: F401
    LIB_PATH,
    PDA_ERR_CUDA,
    PDA_ERR_DEVICE_TIMEOUT,
    PDA_ERR_INVALID_ARG,
    PDA_ERR_NOALLOC_CAPACITY,
    PDA_ERR_UNSUPPORTED,
    PDA_ERR_WORKSPACE,
    KERNEL_NAMES,
    PDA_KERNEL_PER_UNIT,
    PDA_KERNEL_PER_UNIT_DENSE,
    PDA_KERNEL_PERSISTENT,
    PDA_KV_NATIVE,
    PDA_KV_SHUFFLED_V,
    PDA_OK,
    PDA_OUT_BF16,
    PDA_OUT_E4M3,
    PdaError,
    choose_kernel,
    choose_splits,
    decode,
    decode_ex,
    decode_host,
    decode_noalloc,
    decode_slot_scales,
    decode_strided,
    decode_raw,
    load,
    plan_kernel,
    plan_launches,
    plan_slot_scales,
    tail_pieces,
    plan_splits,
    query_device_status,
    workspace_info,
    release,
    reserve,
    reshape_and_cache,
    set_block_check,
    set_profile_events,
    set_split_override,
    set_tail_split,
    set_tma_gather,
    status_string,
    bounded_wait_check,
)
