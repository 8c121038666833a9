"""Seeded synthetic inputs for the decode path (shared by tests, bench and smoke).

This module only draws random numbers in the shapes and distributions of the
workloads; it holds none of the method's arithmetic (no unpacking, no
dequantisation, no norms, no attention).  Both the CUDA path and the CPU
oracle receive the arrays it returns.

Distributions (the pages give none; these follow the workload descriptions):
  * packed int4 weights, layout [N][K/8], one of two code distributions:
      - "full": uniform random uint32 words, so every nibble, hence every
        code in [-8, 7], is equally likely (the single-layer workloads);
      - "symmetric": codes uniform on [-7, 7], what a symmetric quantiser
        with scale amax/7 emits (the multi-layer model workloads: the
        [-8, 7] codes have mean -1/2, which adds the same offset to every
        GEMV output and overflows fp16 after a few random layers);
  * group scales: fp16, uniform in [0.005, 0.02], layout [N][K/128];
  * activations, embeddings, KV pages: fp16 N(0, 1);
  * RMSNorm gammas: fp16 1 + 0.1 N(0, 1);
  * q/k/v biases: fp16 N(0, 0.1) (omitted for the tiny layer);
  * lm_head: fp16 N(0, 0.02);
  * block tables: distinct pages drawn at random from the pool, entries past
    a sequence's last page set to -1 (never read).
"""
from __future__ import annotations

import numpy as np

PAGE = 16
GROUP = 128

# Workload shapes.  Names say what they are.
TINY_LAYER = dict(name="tiny-layer-h896-ctx37", hidden=896, n_q_heads=7, n_kv_heads=1, head_dim=128,
                  inter=2432, n_layers=1, vocab=0, eps=1e-6, theta=1e6, batch=1, context=37,
                  pool_pages=8, bias=False, seed=1000)
QWEN_LAYER = dict(name="qwen2.5-7b-layer-b1-ctx512", hidden=3584, n_q_heads=28, n_kv_heads=4,
                  head_dim=128, inter=18944, n_layers=1, vocab=0, eps=1e-6, theta=1e6, batch=1,
                  context=512, pool_pages=4096, bias=True, seed=1001)
QWEN_MODEL = dict(name="qwen2.5-7b-28L-b1-ctx512", hidden=3584, n_q_heads=28, n_kv_heads=4,
                  head_dim=128, inter=18944, n_layers=28, vocab=152064, eps=1e-6, theta=1e6, batch=1,
                  context=512, gen_tokens=128, bias=True, codes="symmetric", seed=1002)
QWEN_BATCHED = dict(name="qwen2.5-7b-28L-b32-ctxU1..4096", hidden=3584, n_q_heads=28, n_kv_heads=4,
                    head_dim=128, inter=18944, n_layers=28, vocab=152064, eps=1e-6, theta=1e6, batch=32,
                    max_context=4096, forced_lens=(15, 16, 17), pool_pages=16384, bias=True, codes="symmetric",
                    seed=1003)
QWEN_LONG = dict(name="qwen2.5-7b-layer-b4-ctx32768", hidden=3584, n_q_heads=28, n_kv_heads=4,
                 head_dim=128, inter=18944, n_layers=1, vocab=0, eps=1e-6, theta=1e6, batch=4,
                 context=32768, pool_pages=16384, partition_tokens=512, bias=True, seed=1004)


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


# The 225 byte values whose two nibbles are both non-zero (no code -8).
_BYTES_NO_ZERO_NIBBLE = np.array([b for b in range(256) if (b & 0xF) and (b >> 4)], dtype=np.uint8)


def int4_weight(r: np.random.Generator, N: int, K: int, codes: str = "full"):
    """(qweight uint32 [N][K/8], scales fp16 [N][K/128])."""
    assert K % GROUP == 0
    if codes == "full":
        qw = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    elif codes == "symmetric":
        idx = r.integers(0, len(_BYTES_NO_ZERO_NIBBLE), size=(N, K // 2), dtype=np.uint8)
        qw = np.ascontiguousarray(_BYTES_NO_ZERO_NIBBLE[idx]).view("<u4").reshape(N, K // 8)
    else:
        raise ValueError(codes)
    s = r.uniform(0.005, 0.02, size=(N, K // GROUP)).astype(np.float16)
    return qw, s


def normal_fp16(r: np.random.Generator, shape, std: float = 1.0, mean: float = 0.0):
    return (r.standard_normal(shape, dtype=np.float32) * np.float32(std) + np.float32(mean)).astype(np.float16)


def gamma(r: np.random.Generator, H: int):
    return normal_fp16(r, (H,), std=0.1, mean=1.0)


def layer_weights(r: np.random.Generator, cfg: dict) -> dict:
    H, Hq, Hkv, D, I = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["inter"]
    w = {"ln1": gamma(r, H), "ln2": gamma(r, H)}
    codes = cfg.get("codes", "full")
    for name, N, K in (("q", Hq * D, H), ("k", Hkv * D, H), ("v", Hkv * D, H), ("o", H, Hq * D),
                       ("g", I, H), ("u", I, H), ("d", H, I)):
        w["w" + name], w["s" + name] = int4_weight(r, N, K, codes)
    if cfg.get("bias", False):
        w["bq"] = normal_fp16(r, (Hq * D,), 0.1)
        w["bk"] = normal_fp16(r, (Hkv * D,), 0.1)
        w["bv"] = normal_fp16(r, (Hkv * D,), 0.1)
    else:
        w["bq"] = w["bk"] = w["bv"] = None
    return w


def kv_pool(r: np.random.Generator, pages: int, Hkv: int, D: int):
    """fp16 N(0,1) pool, layout [pages][Hkv][16][D]."""
    return normal_fp16(r, (pages, Hkv, PAGE, D))


def block_table(r: np.random.Generator, lens, pool_pages: int, max_blocks: int | None = None):
    """Disjoint random pages for each sequence; -1 past each sequence's need."""
    lens = [int(x) for x in lens]
    need = [(L + PAGE - 1) // PAGE for L in lens]
    if max_blocks is None:
        max_blocks = max(1, max(need))
    assert sum(need) <= pool_pages
    perm = r.permutation(pool_pages).astype(np.int32)
    bt = np.full((len(lens), max_blocks), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    return bt


def batched_lens(r: np.random.Generator, B: int, max_context: int, forced=(15, 16, 17)):
    lens = r.integers(1, max_context + 1, size=B).astype(np.int32)
    for i, L in enumerate(forced):
        lens[i] = L
    return lens


def layer_case(cfg: dict, lens=None, seed: int | None = None) -> dict:
    """One decoder layer's weights, input, pools and paging state."""
    r = rng(cfg["seed"] if seed is None else seed)
    B = cfg["batch"]
    w = layer_weights(r, cfg)
    x = normal_fp16(r, (B, cfg["hidden"]))
    if lens is None:
        lens = np.full(B, cfg["context"], np.int32)
    lens = np.asarray(lens, np.int32)
    pool_pages = cfg["pool_pages"]
    k_pool = kv_pool(r, pool_pages, cfg["n_kv_heads"], cfg["head_dim"])
    v_pool = kv_pool(r, pool_pages, cfg["n_kv_heads"], cfg["head_dim"])
    bt = block_table(r, lens, pool_pages)
    return dict(weights=w, x=x, k_pool=k_pool, v_pool=v_pool, block_table=bt, context_lens=lens)


def model_case(cfg: dict, lens, gen_tokens: int = 0, pool_pages: int | None = None, seed: int | None = None) -> dict:
    """Whole-model inputs for B = len(lens) sequences.

    lens[b] tokens of KV are already cached for sequence b (0 is allowed);
    each block table also covers gen_tokens further positions, so the pages
    of the tokens still to be decoded are assigned up front.  Only the pages
    some table names carry data (N(0,1), drawn per layer into k_used / v_used,
    rows in the order of used_pages); the rest of each pool is zero and is
    never read.  host_pool() expands one layer's pool to its full
    [pool_pages][Hkv][16][D] layout."""
    r = rng(cfg["seed"] if seed is None else seed)
    L, H, Hkv, D, V = cfg["n_layers"], cfg["hidden"], cfg["n_kv_heads"], cfg["head_dim"], cfg["vocab"]
    layers = [layer_weights(r, cfg) for _ in range(L)]
    lens = np.asarray(lens, np.int32)
    pool_pages = int(pool_pages or cfg.get("pool_pages", 256))
    bt = block_table(r, lens + gen_tokens, pool_pages)
    used = np.unique(bt[bt >= 0]).astype(np.int64)
    k_used = [normal_fp16(r, (len(used), Hkv, PAGE, D)) for _ in range(L)]
    v_used = [normal_fp16(r, (len(used), Hkv, PAGE, D)) for _ in range(L)]
    embed = normal_fp16(r, (V, H))
    fnorm = gamma(r, H)
    lm = normal_fp16(r, (V, H), std=0.02)
    tok = r.integers(0, V, size=len(lens)).astype(np.int32)
    return dict(cfg=cfg, layers=layers, k_used=k_used, v_used=v_used, used_pages=used, pool_pages=pool_pages,
                bt=bt, lens=lens, tok=tok, embed=embed, fnorm=fnorm, lm=lm)


def host_pool(case: dict, layer: int, which: str) -> np.ndarray:
    """Layer `layer`'s K (which="k") or V ("v") pool as one numpy array."""
    cfg = case["cfg"]
    p = np.zeros((case["pool_pages"], cfg["n_kv_heads"], PAGE, cfg["head_dim"]), np.float16)
    p[case["used_pages"]] = case[which + "_used"][layer]
    return p
