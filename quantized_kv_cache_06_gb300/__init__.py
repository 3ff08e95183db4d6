"""GB300-native TurboQuant packed KV cache: row writer and paged decode attention.

The compute lives in libtq_gb300.so (hand-written CUDA for sm_103a, C ABI in
include/tq.h).  This package is its thin Python binding; it loads the library on
first use and raises if it has not been built.
"""

from ._lib import (  # noqa: F401
    TQ_ERR_BLOCK_OUT_OF_RANGE,
    TQ_ERR_CUDA,
    TQ_ERR_INVALID_ARG,
    TQ_ERR_SLOT_OUT_OF_RANGE,
    TQ_ERR_TIMEOUT,
    TQ_ERR_UNSUPPORTED,
    TQ_OK,
    TQ_RECIPE_TURBOQUANT25,
    TQ_RECIPE_TURBOQUANT35,
    RecipeCodec,
    TQError,
    lib,
    raise_for_device_status,
    tq_build_qjl_matrix,
    tq_build_rotation,
    tq_codebook,
    tq_dequant_rows,
    tq_launch_count,
    tq_paged_decode,
    tq_paged_decode_prod,
    tq_paged_decode_recipe,
    tq_paged_decode_static,
    tq_paged_decode_workspace,
    tq_paged_prefill,
    tq_paged_prefill_int8q,
    tq_prod_row_bytes,
    tq_quantize_queries_int8,
    tq_recipe_calibrate,
    tq_recipe_channel_order,
    tq_recipe_row_bytes,
    tq_row_bytes,
    tq_set_wait_limit,
    tq_write_kv,
    tq_write_kv_prod,
    tq_write_kv_recipe,
)
