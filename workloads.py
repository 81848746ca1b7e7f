"""Seeded synthetic inputs and workload shapes for the reduce/gather collective.

This module only draws numbers and states sizes.  It holds none of the
collective's arithmetic (no sums, no layout offsets), so that the CPU oracle
and the CUDA library can both take their inputs from it without sharing any
of the computation they are compared on.

Every buffer is returned as a numpy array of the element's raw storage:
bf16 and fp16 as uint16 bits, fp32 as float32, int32 as int32.

Workloads (W = emulated ranks, N = elements per rank):
  SMALL      W=2, bf16, N=4096, uniform[-1, 1]
  LARGE      W=8, bf16, N=2^24 (32 MiB per rank), N(0, 1)
  FSDP_LAYER W=8 (4 per node x 2 nodes), bf16, one transformer layer with
             hidden 3584 / kv 512 / ffn 18944, every weight flattened and
             split evenly into W shards, N(0, 0.02); repeated over 28 layers
  AG_SWEEP   W=8, {bf16, fp16, fp32, int32}, 1 KiB .. 512 MiB per rank in
             powers of two, random bits (int32 uniform over the full range)
  LATENCY    W=8, bf16, 8 KiB .. 256 KiB per rank in powers of two,
             uniform[-1, 1], 1000 back-to-back calls
"""
import numpy as np
import torch

ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp32": 4, "int32": 4}
STORAGE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "int32": np.int32}
TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32,
               "int32": torch.int32}

SMALL = dict(name="W2_bf16_4096", W=2, dtype="bf16", N=4096, dist="uniform", seed_base=1000)
LARGE = dict(name="W8_bf16_2^24", W=8, dtype="bf16", N=1 << 24, dist="normal", seed_base=2000)

# Weight shapes of one transformer layer (rows, cols): q, k, v, o, gate, up, down.
FSDP_LAYER_PARAMS = (
    ("q", 3584, 3584), ("k", 512, 3584), ("v", 512, 3584), ("o", 3584, 3584),
    ("gate", 18944, 3584), ("up", 18944, 3584), ("down", 3584, 18944),
)
FSDP_LAYER = dict(name="fsdp_layer_W8_G4x2_bf16", W=8, G=4, dtype="bf16", layers=28,
                  sigma=0.02, seed_base=3000)
AG_SWEEP = dict(W=8, dtypes=("bf16", "fp16", "fp32", "int32"),
                bytes_per_rank=tuple(1 << k for k in range(10, 30)), seed_base=4000)
LATENCY = dict(W=8, dtype="bf16", bytes_per_rank=tuple(1 << k for k in range(13, 19)),
               calls=1000, seed_base=5000)


def shard_sizes(params, W):
    """E_s per param: each flattened weight split evenly into W shards."""
    out = []
    for _, rows, cols in params:
        n = rows * cols
        if n % W:
            raise ValueError("weights must split evenly over the ranks")
        out.append(n // W)
    return out


def _f32_to_storage(x: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp16":
        return x.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp32":
        return x.numpy().astype(np.float32, copy=False)
    raise ValueError(dtype)


def rank_buffer(n: int, dtype: str, dist: str, seed: int, sigma: float = 1.0) -> np.ndarray:
    """One rank's buffer of n elements.

    dist: "uniform" (U[-1, 1]), "normal" (N(0, sigma)), "bits" (uniform random
    bit patterns: NaN and Inf encodings included), "int" (int32 uniform over
    the full range; the same as "bits" for int32).
    """
    if dist in ("bits", "int") or dtype == "int32":
        rng = np.random.default_rng(seed)
        if ELEM_BYTES[dtype] == 2:
            return rng.integers(0, 1 << 16, size=n, dtype=np.uint16)
        raw = rng.integers(-(1 << 31), 1 << 31, size=n, dtype=np.int32)
        return raw.view(np.float32) if dtype == "fp32" else raw
    g = torch.Generator().manual_seed(seed)
    if dist == "uniform":
        x = torch.rand(n, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn(n, generator=g, dtype=torch.float32) * sigma
    else:
        raise ValueError(dist)
    return _f32_to_storage(x, dtype)


def rank_buffers(W: int, n: int, dtype: str, dist: str, seed_base: int, sigma: float = 1.0):
    """W rank buffers; rank r uses seed seed_base + r."""
    return [rank_buffer(n, dtype, dist, seed_base + r, sigma) for r in range(W)]


def fsdp_layer_shards(W: int, layer: int, sigma: float = 0.02, seed_base: int = 3000,
                      params=FSDP_LAYER_PARAMS):
    """Full flattened weights of one layer and each rank's shard buffer.

    Returns (full_params, shards): full_params[s] is weight s flattened
    (raw storage bits); shards[r] is rank r's FSDP shard, the concatenation
    over s of the r-th equal slice of full_params[s].
    """
    E = shard_sizes(params, W)
    full = [rank_buffer(rows * cols, "bf16", "normal", seed_base + 100 * layer + s, sigma)
            for s, (_, rows, cols) in enumerate(params)]
    shards = [np.concatenate([full[s][r * E[s]:(r + 1) * E[s]] for s in range(len(params))])
              for r in range(W)]
    return full, shards
