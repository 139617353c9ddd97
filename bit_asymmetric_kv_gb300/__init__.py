"""GB300-native (sm_103a) KIVI asymmetric 2-bit KV cache: quantize, stream, decode.

The compute runs in the CUDA library ``lib/libkivi.so`` (C ABI in include/kivi.h);
``bit_asymmetric_kv_gb300.kivi`` is its Python binding and ``synth`` holds the
seeded synthetic workloads.  Import is cheap: the library loads on first use.
"""
from . import synth  # noqa: F401
from .kivi import (Cache, KiviError, PagedCache, kivi_append_token, kivi_buffer_bytes,  # noqa: F401
                   kivi_decode_attention, kivi_decode_splits, kivi_decode_step, kivi_decode_workspace_bytes,
                   kivi_dequantize_debug, kivi_paged_append_token, kivi_paged_buffer_bytes,
                   kivi_paged_decode_attention, kivi_paged_decode_step, kivi_paged_decode_workspace_bytes,
                   kivi_paged_prefill, kivi_quantize_prefill, kivi_status_string, make_dims, make_paged_dims,
                   paged_workspace, workspace)
