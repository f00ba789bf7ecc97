// prefill.cu -- exact attention forward for sm_103a in one tiled pass.
//
// The method: "Capstone: CUDA Softmax 与 Attention 算子", section 4.1 (the
// FlashAttention-2 loop order: a CTA owns query tiles, the inner loop streams
// K/V tiles, O stays on chip and is written once), section 4.2 (unnormalised
// accumulation O <- O * e^(m_old - m_new) + P V with one final division by l)
// and section 2.2 steps 3-5 (the online running max m and denominator l).
// The asynchrony follows the intent of "Flash Attention 3 指南" (the FA3
// sketch: asynchronous tile loads, asynchronous GEMMs, softmax overlapped
// with the next GEMM) and the warp roles of "FlashAttention V3 实战",
// section 2.2 (producer warp for TMA, consumer warps for math and softmax),
// redesigned for Blackwell:
//
//   Persistent CTAs, one per SM.  A work unit is a pair of 128-row query
//   tiles of one (batch, head); units are dealt to CTAs in snake order
//   (longest first for causal masks, head-major otherwise).
//
//   warp 2      TMA producer: Q tile 0 and 1 of each unit, then K_j, V_j of
//               every KV block into an NST-stage shared-memory ring guarded
//               by full/empty mbarrier pairs; runs ahead across units.
//   warp 0, 1   MMA issuers, one thread each, for query tile 0 and 1:
//               tcgen05.mma S_t = Q_t K_j^T into tensor memory, then
//               O_t += P_t V_j with P_t read from tensor memory; completion is
//               signalled with tcgen05.commit.  The two issuers take strict
//               turns so the pipe sees S0(j), PV1(j-1), S1(j), PV0(j) order
//               (each softmax overlaps two GEMMs of the other tile).
//   warps 3-6   softmax for tile 0, warps 7-10 for tile 1: one thread per row
//               reads its S row from tensor memory, masks, updates (m, l),
//               writes P (bf16 or e4m3) back over S, rescales O when the
//               running max moved by more than kTau (log2 units), and runs the
//               epilogue (O / l -> bf16 -> per-warp shared staging -> TMA
//               store; LSE).
//
// Ordering: a tile's MMAs are issued by one thread and complete in issue
// order, so the commit that signals S_t(j) also proves PV_t(j-1) finished;
// the softmax warpgroup may then rescale O_t and overwrite P_t.
//
// Lazy rescaling: the running max used for the exponentials is raised only
// when the new block max exceeds it by more than kTau; O and l share that
// stale max so O / l is unchanged (the merge identity of section 2.2 step 4
// holds for any common reference point), and p stays <= 2^kTau.
#include "kernels.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace attn {

namespace {

constexpr float kTau = 8.0f;  // log2 units; 2^8 = 256 < 448 (e4m3 max)
constexpr float kLn2 = 0.69314718055994530942f;

template <int D, bool FP8>
struct Cfg {
    static constexpr int EB = FP8 ? 1 : 2;         // bytes per input element
    static constexpr int PANEL = 128 / EB;         // elements in one 128-byte row panel
    static constexpr int NPANEL = D / PANEL;       // panels per row
    static constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B
    static constexpr int TILE_BYTES = NPANEL * PANEL_BYTES;
    static constexpr int NST = (D == 128 && !FP8) ? 4 : 8;  // K/V ring stages
    static constexpr int OST_WARP_BYTES = 2 * 32 * 64;      // two 32x32 bf16 staging buffers per warp
    __host__ __device__ static constexpr uint32_t tm_s(int t) { return t ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256u + (t ? (uint32_t)D : 0u); }
    static constexpr uint32_t TM_COLS = 512;
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + 2 * TILE_BYTES;
    static constexpr int OFF_OST = OFF_KV + NST * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_OST + 8 * OST_WARP_BYTES;
    static constexpr int N_BARS = 2 * NST + 16;
    static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // more than half an SM's shared memory: two CTAs never share one SM's
    // tensor memory (each allocates all 512 columns)
    static constexpr int SMEM_BYTES = (SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024);
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(D % PANEL == 0 && D % 64 == 0, "head dim");
};

struct Bars {
    uint64_t* q_full;    // [2]
    uint64_t* q_empty;   // [2]
    uint64_t* kv_full;   // [NST]
    uint64_t* kv_empty;  // [NST], two arrivals (one per issuer)
    uint64_t* s_full;    // [2]
    uint64_t* p_full;    // [2], 128 arrivals
    uint64_t* o_full;    // [2]
    uint64_t* o_empty;   // [2], 128 arrivals
    uint64_t* done;      // [2]
    uint64_t* turn;      // [2], turn[t]: issuer t may issue its next group
};

// One work unit: query tiles [q0[t], q0[t] + rows[t]) of head bh, each
// needing n[t] KV blocks; J = max(n[0], n[1]) blocks are streamed.
struct Unit {
    int bh, J;
    int q0[2], rows[2], n[2];
};

// Number of KV blocks query tile [q0, q0 + rows) needs (0 = nothing visible).
__device__ __forceinline__ int tile_blocks(int q0, int rows, int Nq, int Nk, int causal) {
    if (rows <= 0) return 0;
    const int kv_blocks = (Nk + 127) / 128;
    if (!causal) return kv_blocks;
    const long long last_key = (long long)q0 + rows - 1 + (Nk - Nq);
    if (last_key < 0) return 0;
    const long long nb = last_key / 128 + 1;
    return nb < kv_blocks ? (int)nb : kv_blocks;
}

__device__ __forceinline__ Unit unit_geometry(const PrefillParams& p, int u) {
    Unit g;
    int pair;
    if (p.causal) {  // heaviest (last) pairs first, all heads of a pair adjacent
        pair = p.n_pairs - 1 - u / p.BH;
        g.bh = u % p.BH;
    } else {  // all pairs of one head adjacent: concurrent units share K/V in L2
        pair = u % p.n_pairs;
        g.bh = u / p.n_pairs;
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        g.q0[t] = (2 * pair + t) * 128;
        const int rr = p.Nq - g.q0[t];
        g.rows[t] = rr < 0 ? 0 : (rr > 128 ? 128 : rr);
        g.n[t] = tile_blocks(g.q0[t], g.rows[t], p.Nq, p.Nk, p.causal);
    }
    g.J = g.n[0] > g.n[1] ? g.n[0] : g.n[1];
    return g;
}

// The r-th unit of this CTA in snake order (rounds of gridDim.x units, every
// other round reversed), or -1 when the CTA has no more units.  `round_` is
// advanced past rounds in which this CTA gets nothing.
__device__ __forceinline__ int next_unit(const PrefillParams& p, int& round_) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    for (;;) {
        const long long base = (long long)round_ * G;
        if (base >= p.n_units) return -1;
        const int u = (int)base + ((round_ & 1) ? (G - 1 - c) : c);
        ++round_;
        if (u < p.n_units) return u;
    }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tma_store_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// ---------------------------------------------------------------- producer

template <int D, bool FP8>
__device__ __forceinline__ bool load_kv(const PrefillParams& p, uint8_t* smem, const Bars& b,
                                        volatile int* abort_flag, int& kv_idx, int j, int bh, bool is_v) {
    using C = Cfg<D, FP8>;
    const int slot = kv_idx % C::NST;
    const int round = kv_idx / C::NST;
    if (round > 0 && !wait_bar(&b.kv_empty[slot], (uint32_t)((round - 1) & 1), abort_flag, p.status)) return false;
    bar_arrive_expect_tx(&b.kv_full[slot], C::TILE_BYTES);
    const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
    uint8_t* dst = smem + C::OFF_KV + slot * C::TILE_BYTES;
#pragma unroll
    for (int pn = 0; pn < C::NPANEL; ++pn)
        tma_load_3d(dst + pn * C::PANEL_BYTES, map, &b.kv_full[slot], pn * C::PANEL, j * 128, bh);
    ++kv_idx;
    return true;
}

template <int D, bool FP8>
__device__ void producer_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag) {
    using C = Cfg<D, FP8>;
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    int kv_idx = 0;
    int qcnt[2] = {0, 0};
    int round_ = 0;
    bool ok = true;
    for (int u = next_unit(p, round_); ok && u >= 0; u = next_unit(p, round_)) {
        const Unit g = unit_geometry(p, u);
        for (int j = 0; ok && j < g.J; ++j) {
            ok = load_kv<D, FP8>(p, smem, b, abort_flag, kv_idx, j, g.bh, false) &&
                 load_kv<D, FP8>(p, smem, b, abort_flag, kv_idx, j, g.bh, true);
            if (!ok || j != 0) continue;
            // the unit's first K/V block is in flight; now its query tiles,
            // each as soon as the previous unit's last S MMA released it
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (g.n[t] == 0) continue;
                if (qcnt[t] > 0 &&
                    !wait_bar(&b.q_empty[t], (uint32_t)((qcnt[t] - 1) & 1), abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                bar_arrive_expect_tx(&b.q_full[t], C::TILE_BYTES);
#pragma unroll
                for (int pn = 0; pn < C::NPANEL; ++pn)
                    tma_load_3d(smem + C::OFF_Q + t * C::TILE_BYTES + pn * C::PANEL_BYTES, &p.tm_q, &b.q_full[t],
                                pn * C::PANEL, g.q0[t], g.bh);
                ++qcnt[t];
            }
        }
    }
    // Drain: every copy this thread started must land before the CTA exits.
    for (int t = 0; t < 2; ++t)
        if (qcnt[t] > 0) drain_wait(&b.q_full[t], (uint32_t)((qcnt[t] - 1) & 1), p.status);
    for (int idx = kv_idx - C::NST > 0 ? kv_idx - C::NST : 0; idx < kv_idx; ++idx)
        drain_wait(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), p.status);
}

// ---------------------------------------------------------------- MMA issuers

// MMA issuers: warp t issues query tile t's GEMMs.  The two issuers take
// strict turns through the turn[] barriers, one group of GEMMs per turn, so
// the tensor pipe sees the fixed order
//   S0(0), S1(0), [PV0(0), S0(1)], [PV1(0), S1(1)], [PV0(1), S0(2)], ...
// (each softmax warpgroup works on its S while the pipe runs the other tile's
// group).  A warp performs its own barrier waits (P ready, K/V landed, O
// drained) before it takes its turn, i.e. while the other warp's GEMMs keep
// the pipe busy; the waits of an issuing thread otherwise leave the pipe idle.
// Slots of the K/V ring are released by both issuers (two arrivals); a tile
// that needs no more blocks of the unit releases with a plain arrive.
template <int D, bool FP8>
__device__ void mma_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                         uint32_t tmem, int t) {
    using C = Cfg<D, FP8>;
    const uint32_t sbase = smem_u32(smem);
    const uint64_t q_desc = sdesc_sw128(sbase + C::OFF_Q + (uint32_t)(t * C::TILE_BYTES), 16, 1024);
    const uint32_t kv0 = sbase + C::OFF_KV;
    const uint32_t d_s = tmem + C::tm_s(t), d_o = tmem + C::tm_o(t);
    auto k_desc = [&](int idx) { return sdesc_sw128(kv0 + (uint32_t)((idx % C::NST) * C::TILE_BYTES), 16, 1024); };
    auto v_desc = [&](int idx) {
        return sdesc_sw128(kv0 + (uint32_t)((idx % C::NST) * C::TILE_BYTES), C::PANEL_BYTES, 1024);
    };
    auto wait_full = [&](int idx) {
        return wait_bar(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), abort_flag, p.status);
    };
    int kv_base = 0, qcnt = 0, units = 0, turns = 0;
    uint32_t sblk = 0;
    bool first = (t == 0);  // the very first group of the CTA needs no turn
    // take the turn: wait until the other issuer has issued its previous group
    auto take_turn = [&]() {
        if (first) {
            first = false;
            return true;
        }
        const bool okw = wait_bar(&b.turn[t], (uint32_t)(turns & 1), abort_flag, p.status);
        ++turns;
        return okw;
    };
    // Pass the turn right after this group's last MMA; the commits follow
    // while the other issuer's GEMMs occupy the pipe.
    auto pass_turn = [&]() { bar_arrive(&b.turn[t ^ 1]); };
    int round_ = 0;
    for (int u = next_unit(p, round_); u >= 0; u = next_unit(p, round_)) {
        const Unit g = unit_geometry(p, u);
        const int nt = g.n[t], J = g.J;
        if (J == 0) continue;
        // ---- start group: S_t(0)
        if (nt > 0) {
            if (!wait_bar(&b.q_full[t], (uint32_t)(qcnt & 1), abort_flag, p.status)) return;
            ++qcnt;
        }
        if (!wait_full(kv_base)) return;
        {
            const uint64_t kd = k_desc(kv_base);
            if (!take_turn()) return;
            tc_fence_after();
            if (nt > 0) issue_s<D, FP8>(d_s, q_desc, kd);
            pass_turn();
            if (nt > 0) {
                tc_commit(&b.s_full[t]);
                if (nt == 1) tc_commit(&b.q_empty[t]);
                tc_commit(&b.kv_empty[kv_base % C::NST]);
            } else {
                bar_arrive(&b.kv_empty[kv_base % C::NST]);
            }
        }
        // ---- group j: PV_t(j), S_t(j+1)
        for (int j = 0; j < J; ++j) {
            const int iV = kv_base + 2 * j + 1, iK1 = kv_base + 2 * j + 2;
            const bool act = j < nt, act_next = j + 1 < nt, k1_used = j + 1 < J;
            if (!wait_full(iV)) return;
            if (k1_used && !wait_full(iK1)) return;
            if (act) {
                if (j == 0 && units > 0 &&
                    !wait_bar(&b.o_empty[t], (uint32_t)((units - 1) & 1), abort_flag, p.status))
                    return;
                if (!wait_bar(&b.p_full[t], sblk & 1u, abort_flag, p.status)) return;
            }
            const uint64_t vd = v_desc(iV);
            const uint64_t kd = k_desc(iK1);
            if (!take_turn()) return;
            tc_fence_after();
            if (act) issue_pv<D, FP8>(d_o, d_s, vd, j > 0);
            if (act_next) issue_s<D, FP8>(d_s, q_desc, kd);
            pass_turn();
            // releases and completions (each commit also covers every earlier MMA of this thread)
            if (act) {
                if (j == nt - 1) tc_commit(&b.o_full[t]);
                ++sblk;
            }
            if (act_next) {
                tc_commit(&b.s_full[t]);
                if (j + 1 == nt - 1) tc_commit(&b.q_empty[t]);
            }
            if (act || act_next)
                tc_commit(&b.kv_empty[iV % C::NST]);
            else
                bar_arrive(&b.kv_empty[iV % C::NST]);
            if (k1_used) {
                if (act_next)
                    tc_commit(&b.kv_empty[iK1 % C::NST]);
                else
                    bar_arrive(&b.kv_empty[iK1 % C::NST]);
            }
        }
        kv_base += 2 * J;
        units += nt > 0;
    }
}

// ---------------------------------------------------------------- softmax + epilogue

template <int D, bool FP8>
__device__ void softmax_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                             uint32_t tmem, int t, int wq, int lane) {
    using C = Cfg<D, FP8>;
    const int r = wq * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::tm_s(t);
    const uint32_t tO = tmem + lane_off + C::tm_o(t);
    const int off = p.Nk - p.Nq;
    const float cs = p.c_scale;
    uint8_t* ost = smem + C::OFF_OST + (t * 4 + wq) * C::OST_WARP_BYTES;
    const uint32_t ost_u = smem_u32(ost);
    uint32_t sblk = 0, units = 0, nstore = 0;
    int round_ = 0;
    bool ok = true;

    for (int u = next_unit(p, round_); ok && u >= 0; u = next_unit(p, round_)) {
        const Unit g = unit_geometry(p, u);
        const int q0 = g.q0[t], rows = g.rows[t], nt = g.n[t], bh = g.bh;
        if (rows <= 0) continue;  // tile lies entirely past Nq
        const int row = q0 + r;
        const long long limit = (long long)row + off;  // last visible key (causal)
        float m = -INFINITY, l = 0.f;

        for (int it = 0; it < nt; ++it, ++sblk) {
            // every lane of the warp takes the same branch (tcgen05.ld is warp-collective)
            ok = __all_sync(0xffffffffu, wait_bar(&b.s_full[t], sblk & 1u, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            uint32_t s[128];
            tmem_ld32(tS + 0, s);
            tmem_ld32(tS + 32, s + 32);
            tmem_ld32(tS + 64, s + 64);
            tmem_ld32(tS + 96, s + 96);
            tmem_ld_wait();
            reg_after_wait<128>(s);

            const int kbase = it * 128;
            const bool need_mask =
                (kbase + 128 > p.Nk) || (p.causal && (long long)kbase + 127 > (long long)q0 + off);
            if (need_mask) {
                // visible columns of this row: [0, bound), the keys up to
                // min(Nk - 1, limit) (causal) or Nk - 1
                long long last = (long long)p.Nk - 1;
                if (p.causal && limit < last) last = limit;
                long long bl = last - kbase + 1;
                const int bound = bl < 0 ? 0 : (bl > 128 ? 128 : (int)bl);
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= bound) s[c] = __float_as_uint(-INFINITY);
            }
            // row max: eight independent chains of 3-input max
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
            // p = 2^(s * cs - m): packed FMA for the argument, MUFU ex2, packed row sums
            const uint64_t cs2 = f2_pack(cs, cs);
            const uint64_t nm2 = f2_pack(-m_use, -m_use);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
            if (FP8) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float p0, p1, p2, p3;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1])), cs2, nm2),
                              p0, p1);
                    f2_unpack(
                        f2_fma(f2_pack(__uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3])), cs2, nm2),
                        p2, p3);
                    p0 = ex2(p0);
                    p1 = ex2(p1);
                    p2 = ex2(p2);
                    p3 = ex2(p3);
                    acc[i & 3] = f2_add(acc[i & 3], f2_add(f2_pack(p0, p1), f2_pack(p2, p3)));
                    w[i] = pack_e4m3x4(p0, p1, p2, p3);
                }
                tmem_st32(tS, w);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // 32 scores -> 16 packed P words per chunk
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float p0, p1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[32 * q + 2 * i]),
                                                 __uint_as_float(s[32 * q + 2 * i + 1])),
                                         cs2, nm2),
                                  p0, p1);
                        p0 = ex2(p0);
                        p1 = ex2(p1);
                        acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
                        w[i] = pack_bf16(p0, p1);
                    }
                    tmem_st16(tS + 16 * q, w);
                }
            }
            {
                float a0, a1;
                f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
                l += a0 + a1;
            }
            // O_t holds PV_t(it-1) complete (see the file comment); rescale it.
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
            tmem_st_wait();
            tc_fence_before();
            bar_arrive(&b.p_full[t]);
        }
        if (!ok) break;

        // ---- epilogue: O_t -> registers (then release O_t), / l, bf16, staged TMA store
        uint32_t o[D];
        if (nt > 0) {
            ok = __all_sync(0xffffffffu, wait_bar(&b.o_full[t], units & 1u, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(tO + 32 * ch, o + 32 * ch);
            tmem_ld_wait();
            reg_after_wait<D>(o);
            tc_fence_before();
            bar_arrive(&b.o_empty[t]);
            ++units;
        } else {
#pragma unroll
            for (int i = 0; i < D; ++i) o[i] = 0u;
        }
        const float m_use = (m == -INFINITY) ? 0.f : m;
        const float inv = (l > 0.f) ? p.o_scale / l : 0.f;
        const bool warp_rows = q0 + wq * 32 < p.Nq;  // some row of this warp is inside the tensor
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
            const uint32_t buf = ost_u + (nstore & 1u) * 2048u;
            if (lane == 0) tma_store_wait_read1();  // the buffer's previous store has read it
            __syncwarp();
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[i] = pack_bf16(__uint_as_float(o[32 * ch + 2 * i]) * inv,
                                 __uint_as_float(o[32 * ch + 2 * i + 1]) * inv);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                st_shared_v4(buf + (uint32_t)(lane * 64 + i * 16), w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (warp_rows) tma_store_3d(&p.tm_o, ost + (nstore & 1u) * 2048u, ch * 32, q0 + wq * 32, bh);
                tma_store_commit();  // one (possibly empty) group per buffer use keeps the count exact
            }
            ++nstore;
        }
        if (p.lse != nullptr && r < rows)
            p.lse[(size_t)bh * p.Nq + row] = (l > 0.f) ? (m_use + lg2(l)) * kLn2 : -INFINITY;
    }
    if (lane == 0) tma_store_wait_all();
}

// ---------------------------------------------------------------- kernel

template <int D, bool FP8>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
    using C = Cfg<D, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    Bars b;
    b.q_full = bars;
    b.q_empty = bars + 2;
    b.kv_full = bars + 4;
    b.kv_empty = bars + 4 + C::NST;
    b.s_full = bars + 4 + 2 * C::NST;
    b.p_full = b.s_full + 2;
    b.o_full = b.p_full + 2;
    b.o_empty = b.o_full + 2;
    b.done = b.o_empty + 2;
    b.turn = b.done + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

    if (threadIdx.x == 0) *skip = (*(volatile unsigned*)p.status != 0u) ? 1 : 0;
    __syncthreads();
    if (*skip) return;  // an earlier launch gave up: leave the device quiet

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            bar_init(&b.q_full[t], 1);
            bar_init(&b.q_empty[t], 1);
            bar_init(&b.s_full[t], 1);
            bar_init(&b.p_full[t], 128);
            bar_init(&b.o_full[t], 1);
            bar_init(&b.o_empty[t], 128);
            bar_init(&b.done[t], 1);
            bar_init(&b.turn[t], 1);
        }
        for (int s = 0; s < C::NST; ++s) {
            bar_init(&b.kv_full[s], 1);
            bar_init(&b.kv_empty[s], 2);
        }
        *abort_flag = 0;
        bar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp >= 3) {
        // warps 3-6: tile 0, warps 7-10: tile 1; a warp reaches TMEM lanes 32*(warp % 4)..+31
        softmax_role<D, FP8>(p, smem, b, abort_flag, tmem, (warp - 3) >> 2, warp & 3, lane);
    } else if (warp < 2) {
        if (lane == 0) {
            mma_role<D, FP8>(p, smem, b, abort_flag, tmem, warp);
            // every issued MMA must finish before tensor memory is released
            tc_commit(&b.done[warp]);
            drain_wait(&b.done[warp], 0, p.status);
        }
        __syncwarp();
    } else {
        if (lane == 0) producer_role<D, FP8>(p, smem, b, abort_flag);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

template <int D, bool FP8>
cudaError_t launch_one(const PrefillParams& p, int grid, cudaStream_t stream) {
    using C = Cfg<D, FP8>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prefill_kernel<D, FP8><<<grid, kPrefillThreads, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

int prefill_smem_bytes(int d, bool fp8) {
    if (fp8) return d == 128 ? Cfg<128, true>::SMEM_BYTES : -1;
    if (d == 128) return Cfg<128, false>::SMEM_BYTES;
    if (d == 64) return Cfg<64, false>::SMEM_BYTES;
    return -1;
}

cudaError_t launch_prefill(int d, bool fp8, const PrefillParams& p, int grid, cudaStream_t stream) {
    if (fp8) {
        if (d == 128) return launch_one<128, true>(p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (d == 128) return launch_one<128, false>(p, grid, stream);
    if (d == 64) return launch_one<64, false>(p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
