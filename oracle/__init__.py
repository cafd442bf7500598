"""CPU oracle of the Prox sparse SwiGLU FFN path. Test infrastructure only: the tests, the
smoke check and the benchmark's CPU-baseline leg may import it; the product path may not."""
from .prox_oracle import *  # noqa: F401,F403
from .prox_oracle import (GROUP, OracleLayer, batch_union, channel_mask, dense_ffn, ffn_batch,
                          ffn_token, k_for, prepare_layer, proxy_accumulators, proxy_salience,
                          proxy_storage_bytes, quantize_activations, quantize_weight_proxy,
                          rmsnorm, select_inputs, silu, stage1_token, stage2_exact)
from .sparsity_allocation import allocate_sparsity, byte_cost_model, normalized_cost

__all__ = ["GROUP", "OracleLayer", "batch_union", "channel_mask", "dense_ffn", "ffn_batch",
           "ffn_token", "k_for", "prepare_layer", "proxy_accumulators", "proxy_salience",
           "proxy_storage_bytes", "quantize_activations", "quantize_weight_proxy", "rmsnorm",
           "select_inputs", "silu", "stage1_token", "stage2_exact", "allocate_sparsity",
           "byte_cost_model", "normalized_cost"]
