"""KV-cache size accounting (test infrastructure; see ``oracle/__init__``).

Follows the tutorial page "LLM 推理服务引擎深度拆解", section 1.3 (KV cache
bytes = 2 for K and V x layers x kv_heads x head_dim x seq_len x dtype_bytes
x batch) and section 5.4 (bytes moved when a request's KV is handed from a
prefill instance to a decode instance: the same product for one request).
The essay page "LLM推理PD分离架构深度工程实践", section 3, works the same
formula per token and per layer.
"""


def kv_cache_bytes(layers: int, kv_heads: int, head_dim: int, seq_len: int,
                   dtype_bytes: int = 2, batch: int = 1) -> int:
    return 2 * layers * kv_heads * head_dim * seq_len * dtype_bytes * batch


def pd_transfer_bytes(seq_len: int, layers: int, kv_heads: int, head_dim: int,
                      dtype_bytes: int) -> int:
    return kv_cache_bytes(layers, kv_heads, head_dim, seq_len, dtype_bytes, 1)


def concurrency_limit(kv_gb_per_request: float, weights_gb: float, total_gb: float,
                      reserve_gb: float = 4.0) -> int:
    """Requests whose KV fits beside the weights and a reserve for activations
    and fragmentation (tutorial page, section 8.1: quantising the KV cache
    raises this limit): floor(free / per-request KV)."""
    free = total_gb - weights_gb - reserve_gb
    return int(free // kv_gb_per_request)
