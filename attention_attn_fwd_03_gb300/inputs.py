"""Seeded synthetic inputs shared by the CUDA path's tests and the oracle.

This module draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both sides of every parity check consume exactly the
tensors produced here.

Recipes (the shapes and distributions of the workloads the attention pages
discuss -- prefill over BHSD tensors and one-token decode over a paged cache):

* dense prefill: a CPU ``torch.Generator`` seeded with ``seed`` draws
  float32 N(0,1) samples for Q, then K, then V, each in [B, H, N, d] order;
  each is rounded to bfloat16 (round-to-nearest-even).
* FP8: the bf16 tensors above, scaled per tensor by s = 448 / amax|X|
  (s = 1 when amax = 0), clamped to +-448 and rounded to float8_e4m3fn;
  descale = 1 / s.  The kernel and the oracle both receive the e4m3 codes and
  the descale.
* paged decode: the CPU generator draws a permutation of the page pool, then
  the per-request lengths (uniform integers in [lo, hi]), then q [B, H, d];
  request r takes the next ceil(len_r / page_size) pages of the permutation,
  unused table entries are -1.  K and V caches [num_pages, page_size, H, d]
  are N(0,1) bf16 drawn by a generator on ``device`` seeded with ``seed``;
  pool pages that no table entry references are filled with NaN so a stray
  read poisons the output.  With grouped KV heads the caches hold H_kv heads
  ([num_pages, page_size, H_kv, d]) and everything else is drawn the same way.
* paged prefill chunks: the CPU generator draws the page permutation, then
  per-request new-token counts q_len (uniform in [q_lo, q_hi]), then cached
  prefix lengths (uniform in [ctx_lo, ctx_hi]), then q [total_q, H, d]
  token-major; seq_len = prefix + q_len keys per request, pages assigned in
  request order from the permutation; caches as for paged decode.
* variable-length batch: per-request q_len, then prefixes, then packed q,
  k, v (see varlen_qkv).
"""
import math

import torch

E4M3_MAX = 448.0


def dense_qkv(B, H, Nq, Nk, d, seed=0, device="cpu"):
    """Q [B,H,Nq,d], K, V [B,H,Nk,d] as bfloat16."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def fp8_quantize(x):
    """Per-tensor amax scaling to float8_e4m3fn; returns (codes, descale float)."""
    amax = float(x.detach().abs().max().float().item()) if x.numel() else 0.0
    s = torch.tensor(E4M3_MAX / amax if amax > 0 else 1.0, dtype=torch.float32)
    y = (x.float() * s.to(x.device)).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return y, float(1.0 / s)


def _fill_tables(seq_lens, perm, max_pages, page_size):
    B = seq_lens.shape[0]
    block_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for r in range(B):
        n = int(math.ceil(int(seq_lens[r]) / page_size))
        block_table[r, :n] = perm[cursor:cursor + n].to(torch.int32)
        cursor += n
    return block_table, perm[:cursor].clone()


def _caches(num_pages, page_size, H_kv, d, used, seed, device, nan_fill_unused):
    gd = torch.Generator(device=device).manual_seed(seed)
    shape = (num_pages, page_size, H_kv, d)
    k_cache = torch.randn(shape, generator=gd, device=device, dtype=torch.bfloat16)
    v_cache = torch.randn(shape, generator=gd, device=device, dtype=torch.bfloat16)
    if nan_fill_unused:
        unused = torch.ones(num_pages, dtype=torch.bool)
        unused[used] = False
        idx = torch.nonzero(unused).flatten().to(device)
        if idx.numel():
            k_cache.index_fill_(0, idx, float("nan"))
            v_cache.index_fill_(0, idx, float("nan"))
    return k_cache, v_cache


def paged_kv(B=64, H=32, d=128, page_size=64, max_pages=128, num_pages=8192,
             len_lo=512, len_hi=8192, seed=0, device="cpu", nan_fill_unused=True, H_kv=None):
    """Returns dict(q, k_cache, v_cache, block_table, seq_lens, used_pages)."""
    H_kv = H if H_kv is None else H_kv
    if H_kv < 1 or H % H_kv:
        raise ValueError("H_kv must divide H")
    if B * max_pages > num_pages:
        raise ValueError("page pool smaller than B * max_pages")
    if len_hi > max_pages * page_size or len_lo < 0 or len_lo > len_hi:
        raise ValueError("length range does not fit the block table")
    g = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)
    seq_lens = torch.randint(len_lo, len_hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    q = torch.randn((B, H, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    block_table, used = _fill_tables(seq_lens, perm, max_pages, page_size)
    k_cache, v_cache = _caches(num_pages, page_size, H_kv, d, used, seed, device, nan_fill_unused)
    return dict(q=q.to(device), k_cache=k_cache, v_cache=v_cache,
                block_table=block_table.to(device), seq_lens=seq_lens.to(device), used_pages=used)


def paged_chunks(B=4, H=8, H_kv=2, d=128, page_size=64, max_pages=16, num_pages=128,
                 q_lo=1, q_hi=256, ctx_lo=0, ctx_hi=512, seed=0, device="cpu", nan_fill_unused=True):
    """Prefill chunks appended to cached prefixes over a paged cache.

    Returns dict(q [total_q, H, d], cu_seqlens_q [B+1] int32, q_lens [B],
    seq_lens [B] int32 (prefix + new tokens), block_table, k_cache, v_cache
    [num_pages, page_size, H_kv, d], used_pages, max_q_len).
    """
    if H_kv < 1 or H % H_kv:
        raise ValueError("H_kv must divide H")
    if B * max_pages > num_pages:
        raise ValueError("page pool smaller than B * max_pages")
    if q_lo < 0 or q_lo > q_hi or ctx_lo < 0 or ctx_lo > ctx_hi or q_hi + ctx_hi > max_pages * page_size:
        raise ValueError("length ranges do not fit the block table")
    g = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)
    q_lens = torch.randint(q_lo, q_hi + 1, (B,), generator=g, dtype=torch.int64)
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (B,), generator=g, dtype=torch.int64)
    seq_lens = (ctx + q_lens).to(torch.int32)
    cu = torch.zeros(B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(q_lens, 0)
    total_q = int(cu[-1])
    q = torch.randn((total_q, H, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    block_table, used = _fill_tables(seq_lens, perm, max_pages, page_size)
    k_cache, v_cache = _caches(num_pages, page_size, H_kv, d, used, seed, device, nan_fill_unused)
    return dict(q=q.to(device), cu_seqlens_q=cu.to(torch.int32).to(device), q_lens=q_lens,
                seq_lens=seq_lens.to(device), block_table=block_table.to(device), k_cache=k_cache,
                v_cache=v_cache, used_pages=used, max_q_len=int(q_lens.max()) if B else 0)


def varlen_qkv(B=8, H=8, H_kv=2, d=128, q_lo=1, q_hi=512, ctx_lo=0, ctx_hi=0, seed=0, device="cpu"):
    """Packed variable-length batch: per request q_len uniform in [q_lo, q_hi]
    new tokens and k_len = q_len + a prefix uniform in [ctx_lo, ctx_hi] keys
    (ctx 0: self-attention of packed sequences).  The CPU generator draws
    q_lens, then prefixes, then q [total_q, H, d], k, v [total_k, H_kv, d] as
    float32 N(0,1) rounded to bf16.  Returns dict(q, k, v, cu_seqlens_q,
    cu_seqlens_k, max_q_len, max_k_len)."""
    if H_kv < 1 or H % H_kv:
        raise ValueError("H_kv must divide H")
    g = torch.Generator(device="cpu").manual_seed(seed)
    q_lens = torch.randint(q_lo, q_hi + 1, (B,), generator=g, dtype=torch.int64)
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (B,), generator=g, dtype=torch.int64)
    k_lens = q_lens + ctx
    cu_q = torch.zeros(B + 1, dtype=torch.int64)
    cu_q[1:] = torch.cumsum(q_lens, 0)
    cu_k = torch.zeros(B + 1, dtype=torch.int64)
    cu_k[1:] = torch.cumsum(k_lens, 0)
    q = torch.randn((int(cu_q[-1]), H, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((int(cu_k[-1]), H_kv, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((int(cu_k[-1]), H_kv, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return dict(q=q.to(device), k=k.to(device), v=v.to(device), cu_seqlens_q=cu_q.to(torch.int32).to(device),
                cu_seqlens_k=cu_k.to(torch.int32).to(device), max_q_len=int(q_lens.max()) if B else 0,
                max_k_len=int(k_lens.max()) if B else 0)


def sample_rows(BH, Nq, n_random=4096, tile=128, seed=0):
    """Flattened row ids (bh * Nq + i) for checking a large problem by sampling.

    Every head contributes rows 0..tile-1, the last tile rows, and every
    tile-boundary row (i % tile in {0, tile-1}); n_random further rows are
    drawn uniformly over all heads.  Sorted and unique.
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    per_head = set(range(min(tile, Nq))) | set(range(max(0, Nq - tile), Nq))
    per_head |= {i for i in range(Nq) if i % tile in (0, tile - 1)}
    per_head = torch.tensor(sorted(per_head), dtype=torch.int64)
    heads = torch.arange(BH, dtype=torch.int64)
    rows = (heads[:, None] * Nq + per_head[None, :]).flatten()
    extra = torch.randint(0, BH * Nq, (n_random,), generator=g, dtype=torch.int64)
    return torch.unique(torch.cat([rows, extra])).numpy()
