// paged.cu -- exact attention over a paged KV cache on the tensor cores:
// grouped-query decode and prefill chunks appended to cached prefixes.
//
// The cache is the block-table layout of "FlashAttention V3 实战: Hopper 架构下
// 的 Paged KV Cache 协同优化", section 3.2 (fixed-size pages named by a
// per-request table, the vLLM / SGLang layout), here with H_kv KV heads per
// slot; query head h reads KV head h / G, G = H / H_kv.  The arithmetic is the
// one-pass online softmax of "Capstone: CUDA Softmax 与 Attention 算子",
// sections 2.2 and 4.1-4.2 (running max m, denominator l, unnormalised O
// rescaled by 2^(m_old - m_new), one final division), in log2 units.
//
// Packing: the G query heads that share a KV head are the rows of one query
// tile, together with up to T = 128 / G consecutive query tokens of the same
// request (row = t * G + g).  Grouped decode thus becomes a [G x d] x [d x 128]
// product per key block that the 128-row tensor-core MMA takes whole, and the
// K/V bytes of a KV head are read once for all G heads.  A prefill chunk
// fills the tile with T tokens.
//
// Work unit = (request, KV head, query tile, split); a split is a run of
// split_blocks KV blocks of 128 keys.  With more than one split the units
// write unnormalised partials (O_s, m_s, l_s) and a merge kernel combines
// them with the (m, l, O) merge of the Capstone page, section 2.2 step 4.
//
// Persistent CTAs (one per SM), 192 threads:
//   warp 0    TMA producer: per unit the Q tile (box: 64 dims x G heads x T
//             tokens), then K_j, V_j of every KV block into an NST-stage ring.
//             A block of 128 keys is gathered from 128 / R page boxes of R
//             rows (R = min(page_size, 128)); the warp's lanes fetch 32 page
//             ids at a time from the block table.  Boxes past the request's
//             keys, or naming an out-of-range page, read the zero fill past
//             the end of the cache.
//   warp 1    MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM S
//             buffers, O += P_j V_j with P_j read from TMEM.  S_{j+1} is issued
//             before PV_j so the next block's scores are computed while the
//             softmax works on the current one.
//   warps 2-5 softmax: one thread per tile row; masks (request length, causal
//             position), updates (m, l) with lazy rescaling (threshold kTau),
//             writes P as bf16 over S, rescales O after PV_{j-1} completed, and
//             zeroes the V rows of a partial last page (cache slots past the
//             request's length may hold anything, and 0 * NaN would poison
//             the P V product); then the epilogue writes O / l (or the
//             partials) and the LSE row by row.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace attn {

namespace {

constexpr float kTau = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct PCfg {
    static constexpr int NPANEL = D / 64;          // 128-byte panels of the head dim
    static constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B
    static constexpr int TILE_BYTES = NPANEL * PANEL_BYTES;
    static constexpr int NST = D == 128 ? 5 : 8;   // K/V ring stages
    static constexpr uint32_t TM_O = 256;          // S buffers at columns 0 and 128
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + TILE_BYTES;
    static constexpr int OFF_BAR = OFF_KV + NST * TILE_BYTES;
    static constexpr int N_BARS = 2 * NST + 9;
    static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // more than half an SM's shared memory: one CTA per SM owns all 512 TMEM columns
    static constexpr int SMEM_BYTES = (SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024);
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct PBars {
    uint64_t* q_full;
    uint64_t* q_empty;
    uint64_t* kv_full;   // [NST]
    uint64_t* kv_empty;  // [NST]
    uint64_t* s_full;    // [2], one per S buffer
    uint64_t* p_full;    // 128 arrivals per block
    uint64_t* o_full;    // one phase per PV product
    uint64_t* o_empty;   // 128 arrivals per unit
    uint64_t* done;
};

struct PUnit {
    int r, kvh, split;
    int q_start, q_len, kv_len;
    int t0, nt;   // the tile's tokens [t0, t0 + nt) of the request; nt <= 0: no tile
    int kb0, nb;  // the unit's KV blocks [kb0, kb0 + nb)
    bool bad;     // the request's offsets or length were out of range
};

// Query tokens and key count of request r, checked against the launch's
// bounds.  Offsets out of range drop the request's queries (q_len = 0); a
// length out of range is clamped.  Either marks the unit bad.
__device__ __forceinline__ void request_extent(const PagedParams& p, int r, PUnit& g) {
    g.bad = false;
    if (p.cu_q != nullptr) {
        const int a = __ldg(p.cu_q + r), b = __ldg(p.cu_q + r + 1);
        g.q_start = a;
        g.q_len = b - a;
        if (a < 0 || b < a || b > p.total_q || g.q_len > p.max_q_len) {
            g.bad = true;
            g.q_start = 0;
            g.q_len = 0;
        }
    } else {
        g.q_start = r;
        g.q_len = 1;
    }
    const int cap = p.max_pages * p.page_size;
    g.kv_len = __ldg(p.seq_lens + r);
    if (g.kv_len < 0 || g.kv_len > cap) {
        g.bad = true;
        g.kv_len = g.kv_len < 0 ? 0 : cap;
    }
}

// KV blocks visible to a tile of a request whose last token is t_last: all
// keys, or under the causal mask the keys up to that token's position
// kv_len - q_len + t_last (bottom-right alignment).
__device__ __forceinline__ int tile_kv_blocks(const PagedParams& p, int q_len, int kv_len, int t_last) {
    long long key_end = kv_len;
    if (p.causal) {
        key_end = (long long)kv_len - q_len + t_last + 1;
        if (key_end > kv_len) key_end = kv_len;
    }
    if (key_end <= 0) return 0;
    return (int)((key_end + 127) / 128);
}

// Unit u: KV head fastest, then request, then query tile (last tiles, the
// heaviest under the causal mask, first), then split.
__device__ __forceinline__ PUnit paged_unit(const PagedParams& p, int u) {
    PUnit g;
    g.kvh = u % p.H_kv;
    int x = u / p.H_kv;
    g.r = x % p.B;
    x /= p.B;
    const int qt = p.n_qt - 1 - x % p.n_qt;
    g.split = x / p.n_qt;
    request_extent(p, g.r, g);
    g.t0 = qt * p.T;
    g.nt = min(p.T, g.q_len - g.t0);
    const int nb_all = g.nt > 0 ? tile_kv_blocks(p, g.q_len, g.kv_len, g.t0 + g.nt - 1) : 0;
    g.kb0 = g.split * p.split_blocks;
    g.nb = max(0, min(p.split_blocks, nb_all - g.kb0));
    return g;
}

__device__ __forceinline__ void st_global_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// ---------------------------------------------------------------- producer (whole warp)

template <int D>
__device__ void producer_role(const PagedParams& p, uint8_t* smem, const PBars& b, volatile int* abort_flag,
                              int lane) {
    using C = PCfg<D>;
    if (lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
    }
    const int R = p.rows_per_box;
    const int LPB = 128 / R;                       // boxes per panel per KV block (1..16)
    const int oob = p.num_pages * p.page_size;     // first row past the cache: zero fill
    int kv_idx = 0, qcnt = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        const PUnit g = paged_unit(p, u);
        if (g.bad && lane == 0) atomicOr(p.status, 1u << kStatusDeviceData);
        if (g.nb == 0) continue;
        // the query tile, once the previous unit's last S product released it
        if (lane == 0) {
            if (qcnt > 0) ok = wait_bar(b.q_empty, (uint32_t)((qcnt - 1) & 1), abort_flag, p.status);
            if (ok) {
                bar_arrive_expect_tx(b.q_full, p.q_tile_bytes);
#pragma unroll
                for (int pn = 0; pn < C::NPANEL; ++pn)
                    tma_load_3d(smem + C::OFF_Q + pn * C::PANEL_BYTES, &p.tm_q, b.q_full, pn * 64, g.kvh * p.G,
                                g.q_start + g.t0);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++qcnt;  // counts issued loads only: the drain below waits for each
        // K and V blocks; lane i holds the cache row of box (batch * 32 + i)
        const long long key0 = (long long)g.kb0 * 128;
        const int n_boxes = g.nb * LPB;
        int my_row = oob;
        for (int j = 0; ok && j < g.nb; ++j) {
            const int box0 = j * LPB;
            if ((box0 & 31) == 0) {
                const int bi = box0 + lane;
                int row = oob;
                if (bi < n_boxes) {
                    const long long key = key0 + (long long)bi * R;
                    if (key < g.kv_len) {
                        const int pg = (int)(key / p.page_size);
                        const int id = __ldg(p.block_table + (size_t)g.r * p.max_pages + pg);
                        if (id >= 0 && id < p.num_pages)
                            row = id * p.page_size + (int)(key % p.page_size);
                        else
                            atomicOr(p.status, 1u << kStatusDeviceData);
                    }
                }
                my_row = row;
            }
            int rows[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) rows[i] = __shfl_sync(0xffffffffu, my_row, (box0 + (i < LPB ? i : 0)) & 31);
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                if (lane == 0) {
                    const int slot = kv_idx % C::NST, round = kv_idx / C::NST;
                    if (round > 0) ok = wait_bar(&b.kv_empty[slot], (uint32_t)((round - 1) & 1), abort_flag, p.status);
                    if (ok) {
                        bar_arrive_expect_tx(&b.kv_full[slot], C::TILE_BYTES);
                        const CUtensorMap* map = kv ? &p.tm_v : &p.tm_k;
                        uint8_t* dst = smem + C::OFF_KV + slot * C::TILE_BYTES;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (i >= LPB) break;
#pragma unroll
                            for (int pn = 0; pn < C::NPANEL; ++pn)
                                tma_load_3d(dst + pn * C::PANEL_BYTES + i * R * 128, map, &b.kv_full[slot], pn * 64,
                                            g.kvh, rows[i]);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                ++kv_idx;
            }
        }
    }
    // Drain: every copy this warp started must land before the CTA exits.
    if (lane == 0) {
        if (qcnt > 0) drain_wait(b.q_full, (uint32_t)((qcnt - 1) & 1), p.status);
        for (int idx = kv_idx - C::NST > 0 ? kv_idx - C::NST : 0; idx < kv_idx; ++idx)
            drain_wait(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), p.status);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- MMA issuer (one thread)

template <int D>
__device__ void mma_role(const PagedParams& p, uint8_t* smem, const PBars& b, volatile int* abort_flag,
                         uint32_t tmem) {
    using C = PCfg<D>;
    const uint32_t sbase = smem_u32(smem);
    const uint64_t q_desc = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
    const uint32_t kv0 = sbase + C::OFF_KV;
    auto k_desc = [&](int idx) { return sdesc_sw128(kv0 + (uint32_t)((idx % C::NST) * C::TILE_BYTES), 16, 1024); };
    auto v_desc = [&](int idx) {
        return sdesc_sw128(kv0 + (uint32_t)((idx % C::NST) * C::TILE_BYTES), C::PANEL_BYTES, 1024);
    };
    auto wait_full = [&](int idx) {
        return wait_bar(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), abort_flag, p.status);
    };
    const uint32_t d_o = tmem + C::TM_O;
    int kv_base = 0, qcnt = 0, units = 0;
    uint32_t sblk = 0;  // KV blocks processed so far: block sblk uses S buffer sblk & 1
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        const PUnit g = paged_unit(p, u);
        const int nb = g.nb;
        if (nb == 0) continue;
        if (!wait_bar(b.q_full, (uint32_t)(qcnt & 1), abort_flag, p.status)) return;
        ++qcnt;
        if (!wait_full(kv_base)) return;
        tc_fence_after();
        issue_s<D, false>(tmem + (sblk & 1u) * 128u, q_desc, k_desc(kv_base));
        tc_commit(&b.s_full[sblk & 1u]);
        tc_commit(&b.kv_empty[kv_base % C::NST]);
        if (nb == 1) tc_commit(b.q_empty);
        for (int j = 0; j < nb; ++j) {
            const uint32_t sb = sblk + (uint32_t)j;
            const int iV = kv_base + 2 * j + 1, iK1 = kv_base + 2 * j + 2;
            if (j + 1 < nb) {  // S_{j+1} into the other buffer (its P_{j-1} was consumed by PV_{j-1})
                if (!wait_full(iK1)) return;
                tc_fence_after();
                issue_s<D, false>(tmem + ((sb + 1u) & 1u) * 128u, q_desc, k_desc(iK1));
                tc_commit(&b.s_full[(sb + 1u) & 1u]);
                tc_commit(&b.kv_empty[iK1 % C::NST]);
                if (j + 1 == nb - 1) tc_commit(b.q_empty);
            }
            if (!wait_full(iV)) return;
            if (j == 0 && units > 0 && !wait_bar(b.o_empty, (uint32_t)((units - 1) & 1), abort_flag, p.status))
                return;
            if (!wait_bar(b.p_full, sb & 1u, abort_flag, p.status)) return;
            tc_fence_after();
            issue_pv<D, false>(d_o, tmem + (sb & 1u) * 128u, v_desc(iV), j > 0);
            tc_commit(b.o_full);
            tc_commit(&b.kv_empty[iV % C::NST]);
        }
        sblk += (uint32_t)nb;
        kv_base += 2 * nb;
        ++units;
    }
}

// ---------------------------------------------------------------- softmax + epilogue

template <int D>
__device__ void softmax_role(const PagedParams& p, uint8_t* smem, const PBars& b, volatile int* abort_flag,
                             uint32_t tmem, int wq, int lane) {
    using C = PCfg<D>;
    const int row = wq * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::TM_O;
    const float cs = p.c_scale;
    const int tr = row / p.G, gh = row % p.G;  // token within the tile, head within the group
    const uint32_t kv_smem = smem_u32(smem + C::OFF_KV);
    uint32_t sblk = 0, ocnt = 0;
    int kv_base = 0;
    bool ok = true;

    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        const PUnit g = paged_unit(p, u);
        if (g.nt <= 0) continue;
        const bool row_ok = tr < g.nt;
        const int head = g.kvh * p.G + gh;
        const size_t grow = (size_t)(g.q_start + g.t0 + (row_ok ? tr : 0)) * p.H + head;  // output row
        if (g.nb == 0) {  // no visible key: O = 0, LSE = -inf (split partials: the merge sees no split)
            if (p.n_splits == 1 && g.split == 0 && row_ok) {
                uint16_t* dst = p.o + grow * D;
#pragma unroll
                for (int c = 0; c < D; c += 8) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
                if (p.lse != nullptr) p.lse[grow] = -INFINITY;
            }
            continue;
        }
        const long long kv_len = g.kv_len;
        const long long pos0 = kv_len - g.q_len + g.t0;  // position of the tile's first token
        const long long limit = (p.causal && row_ok) ? min(kv_len - 1, pos0 + tr) : kv_len - 1;
        const long long tile_limit = p.causal ? min(kv_len - 1, pos0) : kv_len - 1;  // smallest row limit
        float m = -INFINITY, l = 0.f;

        for (int j = 0; j < g.nb; ++j, ++sblk) {
            const uint32_t tS = tmem + lane_off + (sblk & 1u) * 128u;
            ok = __all_sync(0xffffffffu, wait_bar(&b.s_full[sblk & 1u], (sblk >> 1) & 1u, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            uint32_t s[128];
            tmem_ld32(tS + 0, s);
            tmem_ld32(tS + 32, s + 32);
            tmem_ld32(tS + 64, s + 64);
            tmem_ld32(tS + 96, s + 96);
            tmem_ld_wait();
            reg_after_wait<128>(s);

            const long long kbase = (long long)(g.kb0 + j) * 128;
            if (kbase + 127 > tile_limit) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (kbase + c > limit) s[c] = __float_as_uint(-INFINITY);
            }
            float mc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float x = __uint_as_float(s[16 * q]);
#pragma unroll
                for (int i = 1; i < 15; i += 2)
                    x = max3(x, __uint_as_float(s[16 * q + i]), __uint_as_float(s[16 * q + i + 1]));
                mc[q] = fmaxf(x, __uint_as_float(s[16 * q + 15]));
            }
            const float mx = fmaxf(max3(mc[0], mc[1], mc[2]), max3(mc[3], mc[4], max3(mc[5], mc[6], mc[7])));
            const float m_cand = mx * cs;
            float alpha = 1.f;
            bool resc = false;
            if (m_cand > m + kTau) {
                if (m != -INFINITY) {
                    alpha = ex2(m - m_cand);
                    resc = true;
                }
                l *= alpha;
                m = m_cand;
            }
            const float m_use = (m == -INFINITY) ? 0.f : m;
            const uint64_t cs2 = f2_pack(cs, cs);
            const uint64_t nm2 = f2_pack(-m_use, -m_use);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // 32 scores -> 16 packed bf16 P words per chunk
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float p0, p1;
                    f2_unpack(
                        f2_fma(f2_pack(__uint_as_float(s[32 * q + 2 * i]), __uint_as_float(s[32 * q + 2 * i + 1])),
                               cs2, nm2),
                        p0, p1);
                    p0 = ex2(p0);
                    p1 = ex2(p1);
                    acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
                    w[i] = pack_bf16(p0, p1);
                }
                tmem_st16(tS + 16 * q, w);
            }
            {
                float a0, a1;
                f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
                l += a0 + a1;
            }
            if (j > 0) {  // O holds PV_{j-1} once its phase completed; rescale it if the max moved
                ok = __all_sync(0xffffffffu, wait_bar(b.o_full, ocnt & 1u, abort_flag, p.status));
                ++ocnt;
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * ch, o);
                        tmem_ld_wait();
                        reg_after_wait<32>(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + 32 * ch, o);
                    }
                }
            }
            if (kbase + 128 > kv_len) {
                // the block runs past the request's keys: clear those V rows (a partial
                // last page holds arbitrary bytes there; pages past it were zero-filled)
                const int iV = kv_base + 2 * j + 1;
                ok = __all_sync(0xffffffffu, wait_bar(&b.kv_full[iV % C::NST], (uint32_t)((iV / C::NST) & 1),
                                                      abort_flag, p.status));
                if (!ok) break;
                if (kbase + row >= kv_len) {
                    const uint32_t vrow = kv_smem + (uint32_t)((iV % C::NST) * C::TILE_BYTES + row * 128);
#pragma unroll
                    for (int pn = 0; pn < C::NPANEL; ++pn)
#pragma unroll
                        for (int c = 0; c < 128; c += 16) st_shared_zero16(vrow + (uint32_t)(pn * C::PANEL_BYTES + c));
                    fence_async_smem();
                }
            }
            tmem_st_wait();
            tc_fence_before();
            bar_arrive(b.p_full);
        }
        if (!ok) break;
        kv_base += 2 * g.nb;

        // ---- epilogue: O -> registers (then release O), / l, store
        ok = __all_sync(0xffffffffu, wait_bar(b.o_full, ocnt & 1u, abort_flag, p.status));
        ++ocnt;
        if (!ok) break;
        tc_fence_after();
        uint32_t o[D];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(tO + 32 * ch, o + 32 * ch);
        tmem_ld_wait();
        reg_after_wait<D>(o);
        tc_fence_before();
        bar_arrive(b.o_empty);
        if (!row_ok) continue;
        const float m_use = (m == -INFINITY) ? 0.f : m;
        if (p.n_splits == 1) {
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            uint16_t* dst = p.o + grow * D;
#pragma unroll
            for (int c = 0; c < D; c += 8)
                st_global_v4(dst + c, pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv),
                             pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv),
                             pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv),
                             pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv));
            if (p.lse != nullptr) p.lse[grow] = (l > 0.f) ? (m_use + lg2(l)) * kLn2 : -INFINITY;
        } else {
            const size_t rec = grow * (size_t)p.n_splits + (size_t)g.split;
            float* po = p.part_o + rec * D;
#pragma unroll
            for (int c = 0; c < D; c += 4) st_global_v4(po + c, o[c], o[c + 1], o[c + 2], o[c + 3]);
            *reinterpret_cast<float2*>(p.part_ml + rec * 2) = make_float2((l > 0.f) ? m_use : -INFINITY, l);
        }
    }
}

// ---------------------------------------------------------------- kernels

template <int D>
__global__ void __launch_bounds__(kPagedThreads, 1) paged_kernel(const __grid_constant__ PagedParams p) {
    using C = PCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    PBars b;
    b.q_full = bars;
    b.q_empty = bars + 1;
    b.kv_full = bars + 2;
    b.kv_empty = bars + 2 + C::NST;
    b.s_full = bars + 2 + 2 * C::NST;
    b.p_full = b.s_full + 2;
    b.o_full = b.p_full + 1;
    b.o_empty = b.o_full + 1;
    b.done = b.o_empty + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

    if (threadIdx.x == 0) *skip = (*(volatile unsigned*)p.status != 0u) ? 1 : 0;
    __syncthreads();
    if (*skip) return;  // an earlier launch gave up: leave the device quiet

    if (threadIdx.x == 0) {
        bar_init(b.q_full, 1);
        bar_init(b.q_empty, 1);
        for (int s = 0; s < C::NST; ++s) {
            bar_init(&b.kv_full[s], 1);
            bar_init(&b.kv_empty[s], 1);
        }
        bar_init(&b.s_full[0], 1);
        bar_init(&b.s_full[1], 1);
        bar_init(b.p_full, 128);
        bar_init(b.o_full, 1);
        bar_init(b.o_empty, 128);
        bar_init(b.done, 1);
        *abort_flag = 0;
        bar_init_fence();
    }
    if (warp >= 2) {
        // rows of the Q tile that no load writes (G * T < 128, or fewer tokens
        // in the box) must read as zeros, not stale shared memory
        const uint32_t q0 = smem_u32(smem + C::OFF_Q) + (uint32_t)((threadIdx.x - 64) * (C::TILE_BYTES / 128));
#pragma unroll
        for (int c = 0; c < C::TILE_BYTES / 128; c += 16) st_shared_zero16(q0 + (uint32_t)c);
        fence_async_smem();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp >= 2) {
        softmax_role<D>(p, smem, b, abort_flag, tmem, warp & 3, lane);
    } else if (warp == 1) {
        if (lane == 0) {
            mma_role<D>(p, smem, b, abort_flag, tmem);
            tc_commit(b.done);  // every issued MMA finishes before tensor memory is released
            drain_wait(b.done, 0, p.status);
        }
        __syncwarp();
    } else {
        producer_role<D>(p, smem, b, abort_flag, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

// One warp per output row (query token, query head): combine the row's
// splits with the (m, l, O) merge, m = max_s m_s, l = sum_s l_s 2^(m_s - m),
// O = sum_s 2^(m_s - m) O_s / l, and write O (bf16) and the LSE.
template <int D>
__global__ void __launch_bounds__(256) paged_merge_kernel(const PagedParams p) {
    constexpr int PER = D / 32;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (long long)p.total_q * p.H) return;
    const int tok = (int)(gw / p.H);
    int r = tok;
    if (p.cu_q != nullptr) {  // the last request whose first token is <= tok
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.cu_q + mid) <= tok)
                lo = mid;
            else
                hi = mid - 1;
        }
        r = lo;
    }
    PUnit g;
    request_extent(p, r, g);
    const int t = tok - g.q_start;
    if (t < 0 || t >= g.q_len) return;  // token not owned by a valid request (reported by the main kernel)
    const int t0 = (t / p.T) * p.T;
    const int nb = tile_kv_blocks(p, g.q_len, g.kv_len, min(t0 + p.T, g.q_len) - 1);
    const int ns = (nb + p.split_blocks - 1) / p.split_blocks;
    const size_t rec0 = (size_t)gw * p.n_splits;

    float m = -INFINITY;
    for (int s = lane; s < ns; s += 32) m = fmaxf(m, p.part_ml[(rec0 + s) * 2]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    if (m != -INFINITY) {
        for (int s = lane; s < ns; s += 32) {
            const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + (rec0 + s) * 2);
            l += ml.y * ex2(ml.x - m);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);

    float acc[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c) acc[c] = 0.f;
    if (m != -INFINITY) {
        for (int s = 0; s < ns; ++s) {
            const float w = ex2(p.part_ml[(rec0 + s) * 2] - m);
            const float* src = p.part_o + (rec0 + s) * D + lane * PER;
#pragma unroll
            for (int c = 0; c < PER; ++c) acc[c] = fmaf(w, src[c], acc[c]);
        }
    }
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    uint16_t* dst = p.o + (size_t)gw * D + lane * PER;
#pragma unroll
    for (int c = 0; c < PER; c += 2) *reinterpret_cast<uint32_t*>(dst + c) = pack_bf16(acc[c] * inv, acc[c + 1] * inv);
    if (lane == 0 && p.lse != nullptr) p.lse[gw] = (l > 0.f) ? (m + lg2(l)) * kLn2 : -INFINITY;
}

template <int D>
cudaError_t launch_d(const PagedParams& p, int grid, cudaStream_t stream) {
    using C = PCfg<D>;
    cudaError_t e =
        cudaFuncSetAttribute(paged_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    paged_kernel<D><<<grid, kPagedThreads, C::SMEM_BYTES, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.n_splits == 1) return e;
    const long long warps = (long long)p.total_q * p.H;
    paged_merge_kernel<D><<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

PagedPlan paged_plan(int total_q, int max_q_len, int B, int H, int H_kv, int d, int page_size, int max_pages) {
    PagedPlan pl{};
    pl.G = H / H_kv;
    pl.T = 128 / pl.G;
    if (pl.T > max_q_len) pl.T = max_q_len;
    if (pl.T < 1) pl.T = 1;
    pl.n_qt = (max_q_len + pl.T - 1) / pl.T;
    const long long kv_blocks = ((long long)max_pages * page_size + 127) / 128;
    const long long base = (long long)B * H_kv * pl.n_qt;
    // Decode-like launches (one query tile per request) split every request
    // into runs of 8 KV blocks so lengths that differ by 16x still balance
    // over the SMs; multi-tile launches split only when there are too few
    // units to fill the GPU.
    long long sb = 8;
    if (pl.n_qt > 1) {
        const long long want = (1024 + base - 1) / base;  // splits per unit wanted
        sb = (kv_blocks + want - 1) / want;
        if (sb < 8) sb = 8;
    }
    if (sb > kv_blocks) sb = kv_blocks;
    if (sb < 1) sb = 1;
    pl.split_blocks = (int)sb;
    pl.n_splits = (int)((kv_blocks + sb - 1) / sb);
    pl.n_units = base * pl.n_splits;
    if (pl.n_splits > 1) {
        const size_t recs = (size_t)total_q * H * pl.n_splits;
        pl.part_o_bytes = recs * d * sizeof(float);
        pl.part_ml_bytes = recs * 2 * sizeof(float);
        pl.workspace_bytes = (pl.part_o_bytes + 255) / 256 * 256 + pl.part_ml_bytes;
    }
    return pl;
}

int paged_smem_bytes(int d) {
    if (d == 128) return PCfg<128>::SMEM_BYTES;
    if (d == 64) return PCfg<64>::SMEM_BYTES;
    return -1;
}

cudaError_t launch_paged(int d, const PagedParams& p, int grid, cudaStream_t stream) {
    if (d == 128) return launch_d<128>(p, grid, stream);
    if (d == 64) return launch_d<64>(p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
