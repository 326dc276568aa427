"""GB300 paged KV cache hot path: slot mapping, scatter, gather and fused
paged decode attention (bf16, fp32 and int8 pools), paged prefill attention,
block copy / swap and the host block allocator, as hand-written CUDA and C++
behind the C ABI in ``include/pkv.h`` (``libpkv.so``), with this thin ctypes
binding."""

from ._binding import (  # noqa: F401
    Allocator,
    append_tokens,
    Pool,
    PkvError,
    STATUS_CODES,
    build_slot_mapping,
    copy_blocks,
    decode_attention,
    decode_attention_shared_prefix,
    decode_shared_prefix_workspace_size,
    decode_step,
    decode_attention_static,
    decode_workspace_size,
    device_error,
    gather,
    get_validate,
    get_wait_limit_ns,
    int8_row_bytes,
    library_path,
    load,
    prefill_attention,
    set_decode_ctas,
    set_debug_skip_fill,
    set_decode_events,
    set_validate,
    set_wait_limit_ns,
    status_string,
    swap_in,
    swap_out,
    version,
    write_slots,
)
from .build import build  # noqa: F401
