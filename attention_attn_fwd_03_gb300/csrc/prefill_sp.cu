// prefill_sp.cu -- exact attention forward for sm_103a, the decoupled design
// for long rows: S and P handed over separately, so that S of the next block
// is computed while the softmax of the current block still runs.
//
// The method is that of prefill.cu ("Capstone: CUDA Softmax 与 Attention 算子",
// sections 2.2 and 4.1-4.2: FlashAttention-2 loop order, online running max
// m and denominator l, unnormalised accumulation with one final division;
// the asynchrony and warp roles of "Flash Attention 3 指南" and
// "FlashAttention V3 实战", section 2.2), with the same work units (two
// 128-row query tiles of one (batch, head), persistent CTAs in snake order),
// lazy rescaling (kTau) and arithmetic; only the hand-over between the GEMMs
// and the softmax differs:
//
//   warp 2      TMA producer: the unit's two Q tiles, then its K and V blocks
//               into an NST-stage ring, K one block ahead of V (K0, K1, V0,
//               K2, V1, ...: the order the GEMMs consume them).
//   warp 0      S issuer (one thread): S_t(j) = Q_t K_j^T into tensor memory
//               as soon as tile t's softmax has read S_t(j-1) out (s_free[t]).
//   warp 1      PV issuer (one thread): O_t += P_t(j) V_j into tensor memory
//               with P_t(j) read from shared memory, as soon as the softmax
//               has written it (p_full[t]).  The two issuers are independent
//               instruction streams into the tensor pipe.
//   warps 3-6   softmax for tile 0, warps 7-10 for tile 1: one thread per
//               row reads S from tensor memory, masks, updates (m, l), forms
//               P (bf16 or e4m3) in registers, waits until PV_t(j-1) has read
//               P_t (pv_done[t]), writes P_t(j) as a 128-byte-swizzled
//               K-major tile to shared memory, rescales O_t if the running max
//               rose by more than kTau, and runs the epilogue (O / l -> bf16
//               rows stored directly; LSE).  S_t goes back to the S issuer
//               right after it is read -- except for rows that have seen a
//               key: those skip the block's row max and exponentiate against
//               the running max, and S_t is held until the block's sum shows
//               no exponential above 2^64 (bf16) or 2^kTau (e4m3), else the
//               block is redone from S_t with its exact max.
//
// In prefill.cu P overwrites S in tensor memory, so S_t(j+1) can only be
// computed after PV_t(j): the per-block chain S -> softmax -> PV -> S sets
// the pace there.  Here S_t(j+1) runs during softmax_t(j), and the softmax of
// both tiles overlaps the GEMMs.  The cost: two P tiles in shared memory
// (leaving a 3-stage K/V ring for bf16 d = 128) and unit boundaries at which
// both tiles end together.  On GB300 this kernel is the faster one when the
// units are long (many KV blocks per query tile: long prefill, the FP8
// workload) and the slower one for short rows, so the host picks it by the
// mean number of KV blocks per unit (api.cu).
//
// Ordering per tile: PV_t(j-1) complete (pv_done[t]) proves P_t free and O_t
// holding PV_t(j-1), so the lazy rescale of O_t is safe after that wait; the
// PV issuer issues PV_t(j) only after P_t(j) is written (p_full[t]).
#include "kernels.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace attn {

namespace {

constexpr float kTau = 8.0f;  // log2 units; 2^8 = 256 < 448 (e4m3 max)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kHeadGroup = 4;  // causal unit order: heads streamed together (see unit_geometry)

template <int D, bool FP8>
struct Cfg {
    static constexpr int EB = FP8 ? 1 : 2;         // bytes per input element
    static constexpr int PANEL = 128 / EB;         // elements in one 128-byte row panel
    static constexpr int NPANEL = D / PANEL;       // panels per row
    static constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B
    static constexpr int TILE_BYTES = NPANEL * PANEL_BYTES;
    static constexpr int P_PANELS = EB;            // 128 keys x EB bytes per P row, in 128-byte panels
    static constexpr int P_BYTES = P_PANELS * PANEL_BYTES;
    // K/V ring stages: what is left of the shared memory after Q and P
    static constexpr int NST = (D == 128 && !FP8) ? 3 : 8;
    __host__ __device__ static constexpr uint32_t tm_s(int t) { return t ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256u + (t ? (uint32_t)D : 0u); }
    static constexpr uint32_t TM_COLS = 512;
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_P = OFF_Q + 2 * TILE_BYTES;  // P tiles of query tile 0 and 1
    static constexpr int OFF_KV = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_BAR = OFF_KV + NST * TILE_BYTES;
    static constexpr int N_BARS = 2 * NST + 20;
    static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // more than half an SM's shared memory: two CTAs never share one SM's
    // tensor memory (each allocates all 512 columns)
    static constexpr int SMEM_BYTES = (SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024);
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(D % PANEL == 0 && D % 64 == 0, "head dim");
};

// Position of each K and V block of a unit in the producer's load order
// K0, K1, V0, K2, V1, ..., K(J-1), V(J-2), V(J-1) (2J loads per unit).
__device__ __forceinline__ int k_load(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_load(int j, int J) { return j == J - 1 ? 2 * J - 1 : 2 * j + 2; }
// Load i of a unit: the block it carries, and whether it is V.
__device__ __forceinline__ int load_block(int i, int J, bool& is_v) {
    if (i == 0) {
        is_v = false;
        return 0;
    }
    if (i == 2 * J - 1) {
        is_v = true;
        return J - 1;
    }
    const int m = i - 1;
    is_v = (m & 1) != 0;
    return is_v ? (m >> 1) : (m >> 1) + 1;
}

struct Bars {
    uint64_t* q_full;    // [2]
    uint64_t* q_empty;   // [2]
    uint64_t* kv_full;   // [NST]
    uint64_t* kv_empty;  // [NST], one arrival (the issuer that read the slot)
    uint64_t* s_full;    // [2], S_t(j) computed (S issuer's commit)
    uint64_t* s_free;    // [2], 128 arrivals: S_t read out of tensor memory
    uint64_t* p_full;    // [2], 128 arrivals: P_t(j) written to shared memory
    uint64_t* pv_done;   // [2], PV_t(j) complete: P_t free, O_t holds PV_t(j)
    uint64_t* o_empty;   // [2], 128 arrivals: O_t read out by the epilogue
    uint64_t* done;      // [2], every MMA of issuer 0 / 1 complete
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
    if (p.causal) {
        // Heads in groups of kHeadGroup; within a group the heaviest (last)
        // pairs first, the group's heads of a pair adjacent.  Concurrent units
        // then stream the K/V of a few heads only, which stays in L2 (measured
        // on 1 x 32 x 32768: DRAM reads 8.6 -> 2.2 GB per launch, and at the
        // power cap the same time for fewer cycles' worth of clock).
        const int hg = p.BH < kHeadGroup ? p.BH : kHeadGroup;
        const int full = p.BH / hg, per = hg * p.n_pairs;
        int gi, r, heads;
        if (u < full * per) {
            gi = u / per;
            r = u - gi * per;
            heads = hg;
        } else {  // the last, smaller group
            gi = full;
            r = u - full * per;
            heads = p.BH - full * hg;
        }
        pair = p.n_pairs - 1 - r / heads;
        g.bh = gi * hg + r % heads;
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
__device__ __forceinline__ int next_unit(int n_units, int& round_) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    for (;;) {
        const long long base = (long long)round_ * G;
        if (base >= n_units) return -1;
        const int u = (int)base + ((round_ & 1) ? (G - 1 - c) : c);
        ++round_;
        if (u < n_units) return u;
    }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}


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
    for (int u = next_unit(p.n_units, round_); ok && u >= 0; u = next_unit(p.n_units, round_)) {
        const Unit g = unit_geometry(p, u);
        // The unit's query tiles first, each as soon as the previous unit's
        // last S MMA released its buffer: Q comes from HBM, as no other unit
        // reads it, so it is the longest load at a unit boundary.
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (g.n[t] == 0) continue;
            if (qcnt[t] > 0 && !wait_bar(&b.q_empty[t], (uint32_t)((qcnt[t] - 1) & 1), abort_flag, p.status)) {
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
        // K0, then K(j+1) ahead of V(j)
        for (int i = 0; ok && i < 2 * g.J; ++i) {
            bool is_v;
            const int j = load_block(i, g.J, is_v);
            ok = load_kv<D, FP8>(p, smem, b, abort_flag, kv_idx, j, g.bh, is_v);
        }
    }
    // Drain: every copy this thread started must land before the CTA exits.
    for (int t = 0; t < 2; ++t)
        if (qcnt[t] > 0) drain_wait(&b.q_full[t], (uint32_t)((qcnt[t] - 1) & 1), p.status);
    for (int idx = kv_idx - C::NST > 0 ? kv_idx - C::NST : 0; idx < kv_idx; ++idx)
        drain_wait(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), p.status);
}

// ---------------------------------------------------------------- MMA issuers

// S issuer (one thread): S_t(j) = Q_t K_j^T for both tiles of every unit,
// block by block.  S_t(j) overwrites S_t(j-1) in tensor memory, so it waits
// until tile t's softmax has read S_t(j-1) out (s_free[t]); it needs the
// unit's Q_t (q_full[t]) and K_j (kv_full).  Commits: s_full[t] per tile,
// q_empty[t] after the tile's last S of the unit, and the K slot.
template <int D, bool FP8>
__device__ void s_issuer_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                              uint32_t tmem) {
    using C = Cfg<D, FP8>;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t kv0 = sbase + C::OFF_KV;
    uint64_t q_desc[2];
    uint32_t d_s[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        q_desc[t] = sdesc_sw128(sbase + C::OFF_Q + (uint32_t)(t * C::TILE_BYTES), 16, 1024);
        d_s[t] = tmem + C::tm_s(t);
    }
    int kv_base = 0, qcnt[2] = {0, 0}, ns[2] = {0, 0};
    int round_ = 0;
    for (int u = next_unit(p.n_units, round_); u >= 0; u = next_unit(p.n_units, round_)) {
        const Unit g = unit_geometry(p, u);
        const int J = g.J;
        for (int j = 0; j < J; ++j) {
            const int iK = kv_base + k_load(j);
            if (!wait_bar(&b.kv_full[iK % C::NST], (uint32_t)((iK / C::NST) & 1), abort_flag, p.status)) return;
            const uint64_t kd = sdesc_sw128(kv0 + (uint32_t)((iK % C::NST) * C::TILE_BYTES), 16, 1024);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (j >= g.n[t]) continue;
                if (j == 0) {
                    if (!wait_bar(&b.q_full[t], (uint32_t)(qcnt[t] & 1), abort_flag, p.status)) return;
                    ++qcnt[t];
                }
                if (ns[t] > 0 && !wait_bar(&b.s_free[t], (uint32_t)((ns[t] - 1) & 1), abort_flag, p.status)) return;
                tc_fence_after();
                issue_s<D, FP8>(d_s[t], q_desc[t], kd);
                ++ns[t];
                tc_commit(&b.s_full[t]);  // before the other tile's S: S_t's softmax starts sooner
                if (j == g.n[t] - 1) tc_commit(&b.q_empty[t]);
            }
            tc_commit(&b.kv_empty[iK % C::NST]);  // j < J: some tile read K_j
        }
        kv_base += 2 * J;
    }
}

// PV issuer (one thread): O_t += P_t(j) V_j for both tiles of every unit,
// block by block, with P_t in shared memory.  Waits for P_t(j) (p_full[t]),
// V_j (kv_full) and, before a unit's first PV_t (which overwrites O_t), for
// the epilogue to have read O_t out (o_empty[t]).  Commits: pv_done[t] per
// PV (P_t free, O_t holds PV_t(j)), and the V slot once both tiles read it.
template <int D, bool FP8>
__device__ void pv_issuer_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                               uint32_t tmem) {
    using C = Cfg<D, FP8>;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t kv0 = sbase + C::OFF_KV;
    uint64_t p_desc[2];
    uint32_t d_o[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        p_desc[t] = sdesc_sw128(sbase + C::OFF_P + (uint32_t)(t * C::P_BYTES), 16, 1024);
        d_o[t] = tmem + C::tm_o(t);
    }
    int kv_base = 0, np[2] = {0, 0}, nu[2] = {0, 0};
    int round_ = 0;
    for (int u = next_unit(p.n_units, round_); u >= 0; u = next_unit(p.n_units, round_)) {
        const Unit g = unit_geometry(p, u);
        const int J = g.J;
        for (int j = 0; j < J; ++j) {
            const int iV = kv_base + v_load(j, J);
            if (!wait_bar(&b.kv_full[iV % C::NST], (uint32_t)((iV / C::NST) & 1), abort_flag, p.status)) return;
            const uint64_t vd = sdesc_sw128(kv0 + (uint32_t)((iV % C::NST) * C::TILE_BYTES), C::PANEL_BYTES, 1024);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (j >= g.n[t]) continue;
                if (!wait_bar(&b.p_full[t], (uint32_t)(np[t] & 1), abort_flag, p.status)) return;
                ++np[t];
                if (j == 0 && nu[t] > 0 &&
                    !wait_bar(&b.o_empty[t], (uint32_t)((nu[t] - 1) & 1), abort_flag, p.status))
                    return;
                tc_fence_after();
                issue_pv_ss<D, FP8>(d_o[t], p_desc[t], vd, j > 0);
                tc_commit(&b.pv_done[t]);
            }
            tc_commit(&b.kv_empty[iV % C::NST]);  // j < J: some tile read V_j
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) nu[t] += g.n[t] > 0;
        kv_base += 2 * J;
    }
}

// ---------------------------------------------------------------- softmax + epilogue

// O_t row *= alpha in tensor memory (rare: the running max rose by more than
// kTau); warp-collective.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
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
    tmem_st_wait();
}

// Store one 16-byte chunk c of row r of a P tile (K-major, 128-byte swizzle:
// chunk position c ^ (r % 8) within the row's 128 bytes, panels of 128 bytes
// of keys PANEL_BYTES apart) -- the layout TMA gives the Q and K tiles.
__device__ __forceinline__ void st_p_chunk(uint32_t p_base, int r, int c, uint32_t a, uint32_t b2, uint32_t c2,
                                           uint32_t d) {
    const uint32_t addr = p_base + (uint32_t)((c >> 3) * (128 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    st_shared_v4(addr, a, b2, c2, d);
}

template <int D, bool FP8>
__device__ void softmax_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                             uint32_t tmem, int t, int wq, int lane) {
    using C = Cfg<D, FP8>;
    constexpr int NW = FP8 ? 32 : 64;  // 32-bit words of one P row
    const int r = wq * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::tm_s(t);
    const uint32_t tO = tmem + lane_off + C::tm_o(t);
    const float cs = p.c_scale;
    const uint32_t p_u = smem_u32(smem + C::OFF_P + t * C::P_BYTES);
    uint32_t ns = 0, npv = 0;
    int round_ = 0;
    bool ok = true;

    for (int u = next_unit(p.n_units, round_); ok && u >= 0; u = next_unit(p.n_units, round_)) {
        const Unit g = unit_geometry(p, u);
        const int q0 = g.q0[t], rows = g.rows[t], nt = g.n[t], bh = g.bh;
        if (rows <= 0) continue;  // tile lies entirely past Nq
        const int Nq_u = p.Nq, Nk_u = p.Nk;
        const int off = Nk_u - Nq_u;
        const int row = q0 + r;
        const long long limit = (long long)row + off;  // last visible key (causal)
        float m = -INFINITY, l = 0.f;

        for (int it = 0; it < nt; ++it, ++ns) {
            // every lane of the warp takes the same branch (tcgen05.ld is warp-collective)
            ok = __all_sync(0xffffffffu, wait_bar(&b.s_full[t], ns & 1u, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            uint32_t s[128];
            auto load_s = [&]() {
                tmem_ld32(tS + 0, s);
                tmem_ld32(tS + 32, s + 32);
                tmem_ld32(tS + 64, s + 64);
                tmem_ld32(tS + 96, s + 96);
                tmem_ld_wait();
                reg_after_wait<128>(s);
            };
            load_s();
            // Rows that have seen a key keep their running max without taking
            // the block's row max.  bf16: P may exceed 1 by far (bf16 and the
            // fp32 sums have 8-bit exponents), so the block stands unless its
            // sum shows an exponential above 2^64.  e4m3 (largest finite 448):
            // it stands if the sum is at most 2^kTau -- then no p exceeds
            // 2^kTau, exactly the case in which the kTau rule would have kept
            // the max, so the result is the same.  S stays in tensor memory
            // until the block stands; otherwise it is redone with its exact max.
            const bool spec = __all_sync(0xffffffffu, m != -INFINITY);
            if (!spec) {
                tc_fence_before();
                bar_arrive(&b.s_free[t]);  // S_t may be overwritten by S_t(it + 1) now
            }

            const int kbase = it * 128;
            const bool need_mask =
                (kbase + 128 > Nk_u) || (p.causal && (long long)kbase + 127 > (long long)q0 + off);
            auto apply_mask = [&]() {
                // visible columns of this row: [0, bound), the keys up to
                // min(Nk - 1, limit) (causal) or Nk - 1
                long long last = (long long)Nk_u - 1;
                if (p.causal && limit < last) last = limit;
                long long bl = last - kbase + 1;
                const int bound = bl < 0 ? 0 : (bl > 128 ? 128 : (int)bl);
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= bound) s[c] = __float_as_uint(-INFINITY);
            };
            float alpha = 1.f;
            bool resc = false;
            auto take_max = [&]() {
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
                if (m_cand > m + kTau) {
                    if (m != -INFINITY) {
                        alpha = ex2(m - m_cand);
                        resc = true;
                    }
                    l *= alpha;
                    m = m_cand;
                }
            };
            if (need_mask) apply_mask();
            if (!spec) take_max();
            // p = 2^(s * cs - m): packed FMA for the argument, MUFU ex2, packed
            // row sums; P packed (bf16 pairs / e4m3 quadruples) into registers
            uint32_t w[NW];
            float lsum;
            auto exps = [&]() {
                const float m_use = (m == -INFINITY) ? 0.f : m;
                const uint64_t cs2 = f2_pack(cs, cs);
                const uint64_t nm2 = f2_pack(-m_use, -m_use);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
                if (FP8) {
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
                } else {  // exponentials over the scores in place; packed once the block is accepted
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        float p0, p1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), cs2, nm2),
                                  p0, p1);
                        p0 = ex2(p0);
                        p1 = ex2(p1);
                        acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
                        s[2 * i] = __float_as_uint(p0);
                        s[2 * i + 1] = __float_as_uint(p1);
                    }
                }
                float a0, a1;
                f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
                lsum = a0 + a1;
            };
            exps();
            if (spec) {
                // bf16: no exponential above 2^64; e4m3: none above 2^kTau = 256 (below its 448)
                if (__any_sync(0xffffffffu, !(lsum <= (FP8 ? 256.f : 0x1p64f)))) {
                    load_s();
                    if (need_mask) apply_mask();
                    take_max();
                    exps();
                }
                tc_fence_before();
                bar_arrive(&b.s_free[t]);  // S_t may be overwritten by S_t(it + 1) now
            }
            l += lsum;
            if (!FP8) {
#pragma unroll
                for (int i = 0; i < 64; ++i) w[i] = pack_bf16(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
            }
            // PV_t(it - 1) has read P_t and O_t holds it complete (the unit's
            // first block: the epilogue of the previous unit waited for its last
            // PV_t), so P_t may be overwritten and O_t rescaled
            if (it > 0) {
                ok = __all_sync(0xffffffffu,
                                wait_bar(&b.pv_done[t], (npv + (uint32_t)it - 1u) & 1u, abort_flag, p.status));
                if (!ok) break;
                tc_fence_after();
            }
#pragma unroll
            for (int c = 0; c < NW / 4; ++c) st_p_chunk(p_u, r, c, w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            if (__any_sync(0xffffffffu, resc)) rescale_o<D>(tO, alpha);  // O_t to the raised max
            fence_async_smem();  // P visible to the tensor core (async proxy)
            tc_fence_before();
            bar_arrive(&b.p_full[t]);
        }
        if (!ok) break;

        // ---- epilogue: O_t -> registers (then release O_t), / l, bf16, row stores
        uint32_t o[D];
        if (nt > 0) {
            ok = __all_sync(0xffffffffu,
                            wait_bar(&b.pv_done[t], (npv + (uint32_t)nt - 1u) & 1u, abort_flag, p.status));
            if (!ok) break;
            npv += (uint32_t)nt;
            tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(tO + 32 * ch, o + 32 * ch);
            tmem_ld_wait();
            reg_after_wait<D>(o);
            tc_fence_before();
            bar_arrive(&b.o_empty[t]);
        } else {
#pragma unroll
            for (int i = 0; i < D; ++i) o[i] = 0u;
        }
        const float m_use = (m == -INFINITY) ? 0.f : m;
        const float inv = (l > 0.f) ? p.o_scale / l : 0.f;
        if (r < rows) {
            const size_t orow = (size_t)bh * p.Nq + row;
            uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c)
                dst[c] = make_uint4(pack_bf16(__uint_as_float(o[8 * c]) * inv, __uint_as_float(o[8 * c + 1]) * inv),
                                    pack_bf16(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv),
                                    pack_bf16(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv),
                                    pack_bf16(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv));
            if (p.lse != nullptr) p.lse[orow] = (l > 0.f) ? (m_use + lg2(l)) * kLn2 : -INFINITY;
        }
    }
}

// ---------------------------------------------------------------- kernel

template <int D, bool FP8>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_sp_kernel(const __grid_constant__ PrefillParams p) {
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
    b.s_free = b.s_full + 2;
    b.p_full = b.s_free + 2;
    b.pv_done = b.p_full + 2;
    b.o_empty = b.pv_done + 2;
    b.done = b.o_empty + 2;
    static_assert(4 + 2 * Cfg<D, FP8>::NST + 12 <= Cfg<D, FP8>::N_BARS, "barrier count");
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

    if (threadIdx.x == 0) *skip = timeout_recorded(p.status) ? 1 : 0;
    __syncthreads();
    if (*skip) return;  // an earlier launch gave up: leave the device quiet

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            bar_init(&b.q_full[t], 1);
            bar_init(&b.q_empty[t], 1);
            bar_init(&b.s_full[t], 1);
            bar_init(&b.s_free[t], 128);
            bar_init(&b.p_full[t], 128);
            bar_init(&b.pv_done[t], 1);
            bar_init(&b.o_empty[t], 128);
            bar_init(&b.done[t], 1);
        }
        for (int s = 0; s < C::NST; ++s) {
            bar_init(&b.kv_full[s], 1);
            bar_init(&b.kv_empty[s], 1);
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
            if (warp == 0)
                s_issuer_role<D, FP8>(p, smem, b, abort_flag, tmem);
            else
                pv_issuer_role<D, FP8>(p, smem, b, abort_flag, tmem);
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
    cudaError_t e =
        cudaFuncSetAttribute(prefill_sp_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prefill_sp_kernel<D, FP8><<<grid, kPrefillThreads, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

int prefill_sp_smem_bytes(int d, bool fp8) {
    if (fp8) return d == 128 ? Cfg<128, true>::SMEM_BYTES : -1;
    if (d == 128) return Cfg<128, false>::SMEM_BYTES;
    if (d == 64) return Cfg<64, false>::SMEM_BYTES;
    return -1;
}

cudaError_t launch_prefill_sp(int d, bool fp8, const PrefillParams& p, int grid, cudaStream_t stream) {
    if (fp8) {
        if (d == 128) return launch_one<128, true>(p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (d == 128) return launch_one<128, false>(p, grid, stream);
    if (d == 64) return launch_one<64, false>(p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
