"""Pins of the float64 oracle against facts fixed by the attention pages and by
mathematics -- never against the oracle's own formula retyped.

Every test here runs on the CPU.  Citations name the page and its section:
  [P3] "Capstone: CUDA Softmax 与 Attention 算子"
  [P2] "FlashAttention V3 实战: Hopper 架构下的 Paged KV Cache 协同优化"
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from attention_attn_fwd_03_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _scores_problem(x):
    """A one-query problem whose scaled scores are exactly x (scale = 1) and
    whose value rows are the identity, so that o equals the probability row."""
    n = len(x)
    q = np.zeros((1, 1, 1, n))
    q[..., 0, 0] = 1.0
    k = np.zeros((1, 1, n, n))
    k[0, 0, :, 0] = x
    v = np.eye(n)[None, None]
    return q, k, v


def _probs_and_lse(x):
    q, k, v = _scores_problem(x)
    o, lse = oracle.attention(q, k, v, scale=1.0)
    return o[0, 0, 0], float(lse[0, 0, 0])


# ---------------------------------------------------------------- worked example

def test_worked_example_two_blocks():
    """[P3] section 2.2 step 3: blocks [1,3] then [2,4] give m=3, l=1.135 after
    the first block and m=4, l=1.553 after the second (printed to 3 decimals)."""
    g = _load("online_softmax_worked_example.json")
    pr = g["printed"]
    tol = 0.5 * 10 ** -g["printed_decimals"] + 1e-12
    a, b = g["block_a"], g["block_b"]
    _, lse_a = _probs_and_lse(a)
    _, lse_b = _probs_and_lse(b)
    p_all, lse_all = _probs_and_lse(a + b)
    m_a, m_b, m_all = max(a), max(b), max(a + b)
    assert m_a == pr["m_a"] and m_all == pr["m_new"] and m_b == pr["m_b"]
    l_a = math.exp(lse_a - m_a)
    l_b = math.exp(lse_b - m_b)
    l_all = math.exp(lse_all - m_all)
    # the page's printed values
    assert abs(l_a - pr["l_a"]) <= tol
    assert abs(l_all - pr["l_new"]) <= tol
    assert abs(l_a * math.exp(m_a - m_all) - pr["l_a_rescaled"]) <= tol
    # the exact closed forms behind them
    assert abs(l_a - (math.exp(-2.0) + 1.0)) < 1e-12
    assert abs(l_all - (math.exp(-3.0) + math.exp(-1.0) + math.exp(-2.0) + 1.0)) < 1e-12
    # [P3] section 2.2 step 4: the merge of the two blocks' (m, l) equals the whole
    m_new = max(m_a, m_b)
    merged = l_a * math.exp(m_a - m_new) + l_b * math.exp(m_b - m_new)
    assert abs(merged - l_all) < 1e-12
    # the probability row is exp(x - m)/l and sums to one
    expect = np.exp(np.array(a + b) - m_all) / l_all
    assert np.max(np.abs(p_all - expect)) < 1e-15
    assert abs(p_all.sum() - 1.0) < 1e-15


def _online_softmax_blocks(x, block):
    """Streaming softmax over blocks (running max and denominator with the
    rescale exp(m_old - m_new)), as [P3] section 2.2 step 4 and section 5
    lab 2 describe; probabilities rebuilt at the end against the final max."""
    m, l = -math.inf, 0.0
    recs = []
    for i in range(0, len(x), block):
        blk = x[i:i + block]
        m_new = max(m, max(blk))
        e = [math.exp(t - m_new) for t in blk]
        l = l * (math.exp(m - m_new) if m != -math.inf else 0.0) + sum(e)
        m = m_new
        recs.append((m_new, e))
    out = []
    for m_blk, e in recs:
        out += [t * math.exp(m_blk - m) / l for t in e]
    return np.array(out), m, l


def test_online_vector_matches_oracle():
    """[P3] section 5 lab 2: the 10-element vector streamed in blocks of 3
    agrees with the three-pass softmax to double-precision accuracy."""
    g = _load("online_softmax_vector.json")
    x = g["vector"]
    p_on, m_on, l_on = _online_softmax_blocks(x, g["block_size"])
    p_or, lse_or = _probs_and_lse(x)
    assert np.max(np.abs(p_on - p_or)) < 1e-15
    assert abs((m_on + math.log(l_on)) - lse_or) < 1e-13


def _fa2_tiled(Q, K, V, Br, Bc):
    """Tiled attention in the FlashAttention-2 order ([P3] section 4.1-4.2):
    Q blocks outside, K/V blocks inside, unnormalised accumulation with the
    exp(m_old - m_new) rescale and one final division by l."""
    N, d = Q.shape
    Nk = K.shape[0]
    scale = 1.0 / math.sqrt(d)
    O = np.zeros_like(Q)
    for i0 in range(0, N, Br):
        Qi = Q[i0:i0 + Br]
        m = np.full((Qi.shape[0], 1), -np.inf)
        l = np.zeros((Qi.shape[0], 1))
        acc = np.zeros((Qi.shape[0], d))
        for j0 in range(0, Nk, Bc):
            S = Qi @ K[j0:j0 + Bc].T * scale
            m_new = np.maximum(m, S.max(axis=1, keepdims=True))
            P = np.exp(S - m_new)
            alpha = np.exp(m - m_new)
            l = l * alpha + P.sum(axis=1, keepdims=True)
            acc = acc * alpha + P @ V[j0:j0 + Bc]
            m = m_new
        O[i0:i0 + Br] = acc / l
    return O


def test_fa2_tiled_equals_oracle():
    """[P3] section 5 lab 3: tiled FA2 (N=64, d=32, Br=Bc=16, numpy seed 42)
    matches plain attention within 1e-10."""
    g = _load("fa2_tiled_demo.json")
    np.random.seed(g["numpy_seed"])
    N, d = g["N"], g["d"]
    Q = np.random.randn(N, d).astype(np.float64)
    K = np.random.randn(N, d).astype(np.float64)
    V = np.random.randn(N, d).astype(np.float64)
    o, _ = oracle.attention(Q[None, None], K[None, None], V[None, None], scale=1.0 / math.sqrt(d))
    t = _fa2_tiled(Q, K, V, g["Br"], g["Bc"])
    assert np.max(np.abs(o[0, 0] - t)) < g["max_abs_err"]


@pytest.mark.parametrize("N,Nk,d,Br,Bc", [(37, 53, 8, 5, 7), (16, 16, 4, 16, 3), (3, 41, 16, 2, 10)])
def test_fa2_tiled_ragged_equals_oracle(N, Nk, d, Br, Bc):
    rng = np.random.default_rng(7)
    Q, K, V = rng.standard_normal((N, d)), rng.standard_normal((Nk, d)), rng.standard_normal((Nk, d))
    o, _ = oracle.attention(Q[None, None], K[None, None], V[None, None], scale=1.0 / math.sqrt(d))
    assert np.max(np.abs(o[0, 0] - _fa2_tiled(Q, K, V, Br, Bc))) < 1e-12


# ---------------------------------------------------------------- closed forms

def _rand(shape, seed, mult=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * mult


def test_zero_query_gives_mean_of_values():
    """Q = 0: every score is 0, so p is uniform over the valid keys:
    o = mean of the valid value rows and lse = ln(n_valid)."""
    B, H, Nq, Nk, d = 2, 3, 5, 11, 8
    q = np.zeros((B, H, Nq, d))
    k, v = _rand((B, H, Nk, d), 1), _rand((B, H, Nk, d), 2)
    o, lse = oracle.attention(q, k, v, scale=0.3)
    assert np.max(np.abs(o - v.mean(axis=2, keepdims=True))) < 1e-14
    assert np.max(np.abs(lse - math.log(Nk))) < 1e-14
    # causal, bottom-right: row i sees keys 0..i+Nk-Nq
    o, lse = oracle.attention(q, k, v, scale=0.3, causal=True)
    for i in range(Nq):
        n = i + Nk - Nq + 1
        assert np.max(np.abs(o[:, :, i] - v[:, :, :n].mean(axis=2))) < 1e-14
        assert np.max(np.abs(lse[:, :, i] - math.log(n))) < 1e-14


def test_constant_values_pass_through():
    """Every value row equal to c gives o = c whatever the scores."""
    B, H, N, d = 1, 2, 9, 6
    q, k = _rand((B, H, N, d), 3, 4.0), _rand((B, H, N, d), 4, 4.0)
    c = _rand((d,), 5)
    v = np.broadcast_to(c, (B, H, N, d)).copy()
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, scale=0.5, causal=causal)
        assert np.max(np.abs(o - c)) < 1e-13


def test_causal_first_row_is_first_value():
    """With Nq == Nk the first query sees only key 0: o_0 = v_0 and lse_0 = s_00."""
    q, k, v = _rand((1, 2, 7, 5), 6), _rand((1, 2, 7, 5), 7), _rand((1, 2, 7, 5), 8)
    scale = 0.37
    o, lse = oracle.attention(q, k, v, scale=scale, causal=True)
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0])) < 1e-15
    s00 = scale * np.einsum("bhc,bhc->bh", q[:, :, 0], k[:, :, 0])
    assert np.max(np.abs(lse[:, :, 0] - s00)) < 1e-14


def test_dominant_score_selects_its_value_row():
    """One score 1000 above all others: p is one-hot up to exp(-1000) = 0 in
    float64, so o equals that value row and lse equals that score."""
    n, d, jstar = 12, 4, 7
    q = np.zeros((1, 1, 1, d)); q[..., 0] = 1.0
    k = np.zeros((1, 1, n, d)); k[0, 0, jstar, 0] = 1000.0
    v = _rand((1, 1, n, d), 9)
    o, lse = oracle.attention(q, k, v, scale=1.0)
    assert np.array_equal(o[0, 0, 0], v[0, 0, jstar])
    assert lse[0, 0, 0] == 1000.0


def test_shift_invariance():
    """Adding c to every score leaves o unchanged and adds c to lse (the
    extra feature column contributes exactly c to each scaled score)."""
    B, H, Nq, Nk, d = 1, 2, 6, 10, 7
    q, k, v = _rand((B, H, Nq, d), 10), _rand((B, H, Nk, d), 11), _rand((B, H, Nk, d), 12)
    scale, c = 0.25, 37.5
    q2 = np.concatenate([q, np.ones((B, H, Nq, 1))], axis=-1)
    k2 = np.concatenate([k, np.full((B, H, Nk, 1), c / scale)], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, Nk, 1))], axis=-1)
    for causal in (False, True):
        o1, l1 = oracle.attention(q, k, v, scale=scale, causal=causal)
        o2, l2 = oracle.attention(q2, k2, v2, scale=scale, causal=causal)
        assert np.max(np.abs(o2[..., :d] - o1)) < 1e-12
        assert np.max(np.abs(l2 - (l1 + c))) < 1e-11


def test_key_permutation_invariance():
    """Without a mask, permuting keys together with their values changes nothing."""
    q, k, v = _rand((2, 2, 5, 8), 13), _rand((2, 2, 19, 8), 14), _rand((2, 2, 19, 8), 15)
    perm = np.random.default_rng(16).permutation(19)
    o1, l1 = oracle.attention(q, k, v, scale=0.4)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], scale=0.4)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13


def test_bounds_and_probability_sums():
    """o is a convex combination of value rows; max_j s_j <= lse <= max_j s_j + ln n;
    each probability row sums to one."""
    B, H, N, d = 2, 2, 33, 16
    q, k, v = _rand((B, H, N, d), 17, 3.0), _rand((B, H, N, d), 18, 3.0), _rand((B, H, N, d), 19)
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o, lse, ps = oracle.attention(q, k, v, scale=scale, causal=causal, with_psum=True)
        assert np.max(np.abs(ps - 1.0)) < 1e-14
        s = scale * np.einsum("bhic,bhjc->bhij", q, k)
        for i in range(N):
            n = i + 1 if causal else N
            smax = s[:, :, i, :n].max(axis=-1)
            assert np.all(lse[:, :, i] >= smax - 1e-12)
            assert np.all(lse[:, :, i] <= smax + math.log(n) + 1e-12)
            lo, hi = v[:, :, :n].min(axis=2), v[:, :, :n].max(axis=2)
            assert np.all(o[:, :, i] >= lo - 1e-12) and np.all(o[:, :, i] <= hi + 1e-12)


def test_causal_rows_equal_truncated_noncausal():
    """Bottom-right causal row i equals the unmasked computation over keys
    0..i+(Nk-Nq); rows with no valid key give o = 0 and lse = -inf."""
    q, k, v = _rand((1, 1, 6, 4), 20), _rand((1, 1, 9, 4), 21), _rand((1, 1, 9, 4), 22)
    o, lse = oracle.attention(q, k, v, scale=0.7, causal=True)
    for i in range(6):
        n = i + 3 + 1
        o_i, l_i = oracle.attention(q[:, :, i:i + 1], k[:, :, :n], v[:, :, :n], scale=0.7)
        assert np.array_equal(o[:, :, i], o_i[:, :, 0]) and np.array_equal(lse[:, :, i], l_i[:, :, 0])
    # more queries than keys: the first Nq-Nk rows have nothing to attend to
    q2 = _rand((1, 1, 8, 4), 23)
    k2, v2 = k[:, :, :5], v[:, :, :5]
    o2, l2 = oracle.attention(q2, k2, v2, scale=0.7, causal=True)
    assert np.all(o2[0, 0, :3] == 0.0) and np.all(np.isneginf(l2[0, 0, :3]))
    assert np.all(np.isfinite(l2[0, 0, 3:]))


def test_row_subset_matches_full():
    q, k, v = _rand((2, 3, 17, 8), 24), _rand((2, 3, 17, 8), 25), _rand((2, 3, 17, 8), 26)
    o, lse = oracle.attention(q, k, v, scale=0.3, causal=True)
    rows = np.array([0, 5, 16, 17, 50, 101])
    o_s, l_s = oracle.attention(q, k, v, scale=0.3, causal=True, rows=rows)
    assert np.array_equal(o_s, o.reshape(-1, 8)[rows]) and np.array_equal(l_s, lse.reshape(-1)[rows])


# ---------------------------------------------------------------- brute force

def _mp_attention(q, k, v, scale, causal):
    import mpmath
    mpmath.mp.dps = 50
    Nq, d = q.shape
    Nk = k.shape[0]
    O = np.zeros((Nq, d)); L = np.zeros(Nq)
    for i in range(Nq):
        n = min(Nk, i + Nk - Nq + 1) if causal else Nk
        s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[i, c]) * mpmath.mpf(k[j, c]) for c in range(d))
             for j in range(n)]
        z = mpmath.fsum(mpmath.exp(t) for t in s)
        for c in range(d):
            O[i, c] = float(mpmath.fsum(mpmath.exp(s[j]) * mpmath.mpf(v[j, c]) for j in range(n)) / z)
        L[i] = float(mpmath.log(z))
    return O, L


@pytest.mark.parametrize("Nq,Nk,d,mult,causal", [(4, 4, 2, 1.0, False), (8, 8, 4, 1.0, True),
                                                  (3, 7, 3, 30.0, False), (6, 8, 4, 30.0, True),
                                                  (1, 1, 1, 1.0, False)])
def test_mpmath_brute_force(Nq, Nk, d, mult, causal):
    """Tiny shapes at 50 digits; N(0,1)*30 scores overflow a softmax that skips
    the max subtraction ([P3] section 6.1), the oracle must stay exact."""
    q, k, v = _rand((Nq, d), 30 + Nq, mult), _rand((Nk, d), 31 + Nk, mult), _rand((Nk, d), 32)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q[None, None], k[None, None], v[None, None], scale=scale, causal=causal)
    O, L = _mp_attention(q, k, v, scale, causal)
    assert np.max(np.abs(o[0, 0] - O)) < 1e-13
    assert np.max(np.abs(lse[0, 0] - L) / np.maximum(1.0, np.abs(L))) < 1e-13


# ---------------------------------------------------------------- element decoding

def test_bf16_decoding_all_codes():
    codes = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    x = codes.view(torch.bfloat16)
    ours = oracle.decode_elems(x)
    ref = x.to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])


def test_e4m3_decoding_all_codes():
    x = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ours = oracle.decode_elems(x)
    ref = x.to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert int(np.isnan(ours).sum()) == 2  # 0x7f and 0xff
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])
    assert np.nanmax(ours) == 448.0


def test_bf16_and_fp8_paths_equal_float64_path():
    """Decoding inside the oracle changes nothing: bf16 (and e4m3 with descales)
    give bit-identical results to passing the widened values as float64."""
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn(1, 2, 9, 8, generator=g).to(torch.bfloat16) for _ in range(3))
    o1, l1 = oracle.attention(q, k, v, scale=0.35, causal=True)
    o2, l2 = oracle.attention(q.double(), k.double(), v.double(), scale=0.35, causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    q8, k8, v8 = (t.float().mul(4).to(torch.float8_e4m3fn) for t in (q, k, v))
    ds = (0.25, 0.5, 0.125)
    o3, l3 = oracle.attention(q8, k8, v8, scale=0.35, descales=ds)
    o4, l4 = oracle.attention(q8.double() * ds[0], k8.double() * ds[1], v8.double() * ds[2], scale=0.35)
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)


# ---------------------------------------------------------------- paged decode

def _small_paged(seed=0, B=5, H=3, d=8, page=4, max_pages=6, num_pages=40):
    from attention_attn_fwd_03_gb300 import inputs
    return inputs.paged_kv(B=B, H=H, d=d, page_size=page, max_pages=max_pages, num_pages=num_pages,
                           len_lo=0, len_hi=page * max_pages, seed=seed)


def test_paged_equals_dense_on_gathered_keys():
    """[P2] section 3.2: key t of request r lives at
    cache[block_table[r][t // page]][t % page]; attention over those keys."""
    p = _small_paged()
    q, kc, vc, bt, sl = p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"]
    o, lse = oracle.paged_decode(q, kc, vc, bt, sl, scale=0.3)
    page = kc.shape[1]
    for r in range(q.shape[0]):
        n = int(sl[r])
        if n == 0:
            assert np.all(o[r] == 0) and np.all(np.isneginf(lse[r]))
            continue
        idx = [(int(bt[r, t // page]), t % page) for t in range(n)]
        kr = torch.stack([kc[a, b] for a, b in idx], dim=1)  # [H, n, d]
        vr = torch.stack([vc[a, b] for a, b in idx], dim=1)
        od, ld = oracle.attention(q[r][:, None, :], kr, vr, scale=0.3)
        assert np.array_equal(o[r], od[:, 0]) and np.array_equal(lse[r], ld[:, 0])
    assert np.all(np.isfinite(o))  # unused pages are NaN and never read


def test_paged_table_invariance():
    """The same logical keys under two different physical page placements give
    the same result."""
    p = _small_paged(seed=1)
    q, kc, vc, bt, sl = p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"]
    o1, l1 = oracle.paged_decode(q, kc, vc, bt, sl, scale=0.3)
    perm = torch.randperm(kc.shape[0], generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm); inv[perm] = torch.arange(perm.numel())
    kc2, vc2 = kc[perm], vc[perm]  # new page i holds old page perm[i]
    bt2 = torch.where(bt >= 0, inv[bt.clamp(min=0).long()].to(torch.int32), bt)
    o2, l2 = oracle.paged_decode(q, kc2, vc2, bt2, sl, scale=0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_bad_page_is_reported():
    p = _small_paged(seed=2)
    bt = p["block_table"].clone()
    r = int(torch.argmax(p["seq_lens"]))
    bt[r, 0] = p["k_cache"].shape[0]  # one past the pool
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(p["q"], p["k_cache"], p["v_cache"], bt, p["seq_lens"], scale=0.3)


# ---------------------------------------------------------------- paged attention: grouped heads, chunks

def _gather(cache, bt, r, n, page):
    """Keys 0..n-1 of request r as [heads, n, d] (test-side gather)."""
    rows = [cache[int(bt[r, t // page]), t % page] for t in range(n)]
    if not rows:
        return cache.new_zeros((cache.shape[2], 0, cache.shape[3]))
    return torch.stack(rows, dim=1)


@pytest.mark.parametrize("H,H_kv", [(8, 2), (8, 1), (6, 3)])
def test_grouped_heads_equal_multihead_on_repeated_cache(H, H_kv):
    """Grouped-query attention is multi-head attention in which the KV head of
    group g serves query heads g*G .. g*G+G-1 (G = H / H_kv): on a cache whose
    heads are repeated G times in that order the two agree exactly.  A head
    map other than h // G (e.g. h % H_kv) fails this."""
    p = inputs.paged_kv(B=5, H=H, d=16, page_size=4, max_pages=6, num_pages=40, len_lo=0, len_hi=24,
                        seed=11, H_kv=H_kv)
    G = H // H_kv
    kc_rep = p["k_cache"].repeat_interleave(G, dim=2)
    vc_rep = p["v_cache"].repeat_interleave(G, dim=2)
    o1, l1 = oracle.paged_attention(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], 0.25)
    o2, l2 = oracle.paged_decode(p["q"], kc_rep, vc_rep, p["block_table"], p["seq_lens"], 0.25)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.all(np.isfinite(o1))


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_chunks_equal_dense_attention_per_request(causal):
    """A prefill chunk of q_len new tokens over seq_len cached keys is dense
    attention with Nq = q_len, Nk = seq_len for each request, with the
    bottom-right causal alignment ([P3] section 7.3's lower-triangular mask
    on the last q_len rows of the full square)."""
    page = 4
    p = inputs.paged_chunks(B=4, H=4, H_kv=2, d=8, page_size=page, max_pages=12, num_pages=60, q_lo=0, q_hi=7,
                            ctx_lo=0, ctx_hi=30, seed=12)
    q, cu, sl, bt = p["q"], p["cu_seqlens_q"], p["seq_lens"], p["block_table"]
    o, lse = oracle.paged_attention(q, p["k_cache"], p["v_cache"], bt, sl, 0.3, cu_seqlens_q=cu, causal=causal)
    G = 2
    for r in range(4):
        a, b = int(cu[r]), int(cu[r + 1])
        if a == b:
            continue
        n = int(sl[r])
        kr = _gather(p["k_cache"], bt, r, n, page).repeat_interleave(G, dim=0)  # [H, n, d]
        vr = _gather(p["v_cache"], bt, r, n, page).repeat_interleave(G, dim=0)
        qd = q[a:b].transpose(0, 1).contiguous()  # [H, q_len, d]
        od, ld = oracle.attention(qd, kr, vr, scale=0.3, causal=causal)
        assert np.array_equal(o[a:b], od.transpose(1, 0, 2)) and np.array_equal(lse[a:b], ld.T)


def test_one_token_per_request_equals_decode():
    """cu_seqlens_q = 0, 1, ..., B with the causal mask: each request's single
    query sits at the last position and sees every cached key."""
    p = inputs.paged_kv(B=6, H=4, d=16, page_size=8, max_pages=4, num_pages=30, len_lo=1, len_hi=32, seed=13)
    cu = torch.arange(7, dtype=torch.int32)
    o1, l1 = oracle.paged_attention(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], 0.2,
                                    cu_seqlens_q=cu, causal=True)
    o2, l2 = oracle.paged_decode(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], 0.2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_zero_query_chunk_gives_prefix_means():
    """Closed form: with q = 0 every visible key has probability 1/n, so under
    the causal mask query i of a request with q_len new tokens over seq_len
    keys returns the mean of the first seq_len - q_len + i + 1 value rows and
    lse = ln(seq_len - q_len + i + 1)."""
    page = 4
    p = inputs.paged_chunks(B=3, H=2, H_kv=1, d=4, page_size=page, max_pages=8, num_pages=30, q_lo=1, q_hi=5,
                            ctx_lo=0, ctx_hi=20, seed=14)
    q = torch.zeros_like(p["q"])
    cu, sl, bt = p["cu_seqlens_q"], p["seq_lens"], p["block_table"]
    o, lse = oracle.paged_attention(q, p["k_cache"], p["v_cache"], bt, sl, 1.0, cu_seqlens_q=cu, causal=True)
    for r in range(3):
        a, b = int(cu[r]), int(cu[r + 1])
        n_len = int(sl[r])
        for i in range(b - a):
            n = n_len - (b - a) + i + 1
            vals = np.array([[float(x) for x in p["v_cache"][int(bt[r, t // page]), t % page, 0]] for t in range(n)])
            for h in range(2):
                assert np.allclose(o[a + i, h], vals.mean(axis=0), rtol=0, atol=1e-14)
                assert abs(lse[a + i, h] - math.log(n)) < 1e-14


def test_paged_attention_rejects_bad_offsets():
    p = inputs.paged_kv(B=2, H=2, d=4, page_size=4, max_pages=2, num_pages=8, len_lo=1, len_hi=8, seed=15)
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(p["q"], p["k_cache"], p["v_cache"], p["block_table"], p["seq_lens"], 1.0,
                               cu_seqlens_q=torch.tensor([0, 2, 1], dtype=torch.int32))


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_dense_attention_per_request(causal):
    """A packed variable-length batch is B independent dense problems; with
    the causal mask each one is aligned bottom-right (k_len >= q_len here,
    and one request with more queries than keys exercises rows that see no
    key)."""
    p = inputs.varlen_qkv(B=5, H=4, H_kv=2, d=8, q_lo=0, q_hi=9, ctx_lo=0, ctx_hi=6, seed=16)
    cu_q, cu_k = p["cu_seqlens_q"].clone(), p["cu_seqlens_k"].clone()
    q, k, v = p["q"], p["k"], p["v"]
    # shrink request 2's keys below its queries (rows with no key under the causal mask)
    r = 2
    qn, kn = int(cu_q[r + 1] - cu_q[r]), int(cu_k[r + 1] - cu_k[r])
    drop = max(0, kn - max(0, qn - 3))
    if drop:
        a = int(cu_k[r + 1]) - drop
        k = torch.cat([k[:a], k[a + drop:]]); v = torch.cat([v[:a], v[a + drop:]])
        cu_k[r + 1:] -= drop
    o, lse = oracle.varlen_attention(q, k, v, cu_q, cu_k, 0.3, causal=causal)
    for rr in range(5):
        a, b = int(cu_q[rr]), int(cu_q[rr + 1])
        ka, kb = int(cu_k[rr]), int(cu_k[rr + 1])
        if a == b:
            continue
        qd = q[a:b].transpose(0, 1).contiguous()
        kd = k[ka:kb].transpose(0, 1).repeat_interleave(2, dim=0).contiguous()
        vd = v[ka:kb].transpose(0, 1).repeat_interleave(2, dim=0).contiguous()
        if kb == ka:
            assert np.all(o[a:b] == 0) and np.all(np.isneginf(lse[a:b]))
            continue
        od, ld = oracle.attention(qd, kd, vd, scale=0.3, causal=causal)
        assert np.array_equal(o[a:b], od.transpose(1, 0, 2)) and np.array_equal(lse[a:b], ld.T)
    if causal:
        assert np.isneginf(lse).any()


# ---------------------------------------------------------------- backward

def _loss(q, k, v, dout, scale, causal):
    o, _ = oracle.attention(q, k, v, scale=scale, causal=causal)
    return float(np.sum(o * dout))


@pytest.mark.parametrize("Nq,Nk,causal", [(3, 5, False), (4, 4, True), (5, 3, True), (2, 6, True)])
def test_backward_equals_finite_differences(Nq, Nk, causal):
    """The gradient of L = sum(dO * O) by central differences of the forward
    oracle (step 1e-5, truncation error ~1e-10) agrees with the backward
    oracle for every element of q, k and v; with Nq > Nk under the causal mask
    some rows see no key and must get zero gradients."""
    rng = np.random.default_rng(Nq * 10 + Nk)
    BH, d, scale = 2, 3, 0.7
    q = rng.standard_normal((BH, Nq, d))
    k = rng.standard_normal((BH, Nk, d))
    v = rng.standard_normal((BH, Nk, d))
    dout = rng.standard_normal((BH, Nq, d))
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, scale, causal=causal)
    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], dout, scale, causal) -
                        _loss(args_m["q"], args_m["k"], args_m["v"], dout, scale, causal)) / (2 * h)
        assert np.allclose(g, num, rtol=0, atol=2e-8), name


def test_backward_identities():
    """Softmax is invariant to a common shift of a row's scores, so every
    row's dS sums to 0 and the dK rows of a head sum to 0; probabilities sum
    to 1, so the dV rows sum to the dO rows; constant value rows make O
    independent of q and k, so dQ = dK = 0."""
    rng = np.random.default_rng(5)
    BH, Nq, Nk, d = 3, 7, 9, 4
    q = rng.standard_normal((BH, Nq, d))
    k = rng.standard_normal((BH, Nk, d))
    v = rng.standard_normal((BH, Nk, d))
    dout = rng.standard_normal((BH, Nq, d))
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, 0.5)
    assert np.allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    assert np.allclose(dv.sum(axis=1), dout.sum(axis=1), atol=1e-12)
    vc = np.broadcast_to(rng.standard_normal((BH, 1, d)), (BH, Nk, d)).copy()
    dq0, dk0, _ = oracle.attention_bwd(q, k, vc, dout, 0.5)
    assert np.allclose(dq0, 0.0, atol=1e-12) and np.allclose(dk0, 0.0, atol=1e-12)


def test_backward_causal_first_row():
    """Under the causal mask query 0 sees only key 0 (p = 1): its dQ is 0 and
    key 0's dV receives all of dO_0."""
    rng = np.random.default_rng(6)
    q, k, v, dout = (rng.standard_normal((1, 4, 3)) for _ in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, 1.0, causal=True)
    assert np.allclose(dq[0, 0], 0.0, atol=1e-14)
    # key 3 is seen only by query 3, key 0 by all four queries
    o, _ = oracle.attention(q, k, v, scale=1.0, causal=True)
    assert np.all(np.isfinite(dv)) and np.allclose(dv.sum(axis=1), dout.sum(axis=1), atol=1e-12)


def test_backward_bf16_inputs_are_decoded_exactly():
    """bf16 inputs give the same gradients as their exact float64 values."""
    q, k, v = inputs.dense_qkv(1, 2, 6, 8, 16, seed=7)
    g = torch.Generator().manual_seed(8)
    dout = torch.randn((1, 2, 6, 16), generator=g).to(torch.bfloat16)
    a = oracle.attention_bwd(q, k, v, dout, 0.25, causal=True)
    b = oracle.attention_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), dout.double().numpy(),
                             0.25, causal=True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_fp8_dequantised_inputs_equal_the_oracle_decoder():
    """The widening the full FP8 workload check does in torch (e4m3 code to
    float64, times the descale, in float64) equals the oracle's own e4m3
    decode times the descale, for every code."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
    finite = torch.isfinite(codes.to(torch.float32))
    desc = 0.0123456789
    ours = (codes.to(torch.float64) * desc)[finite].numpy()
    theirs = (oracle.decode_elems(codes) * desc)[finite.numpy()]
    assert (ours == theirs).all()
