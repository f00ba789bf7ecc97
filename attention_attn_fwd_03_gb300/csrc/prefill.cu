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
//
// Ragged mode (template flag RAGGED, bf16): variable-length sequences of
// token-major tensors, for prefill chunks over a paged cache ("FlashAttention
// V3 实战", section 3.2, the block-table layout) and packed variable-length
// batches.  A schedule pass lists the units (sequence, tile pair, head),
// longest first; the producer warp gathers each key block through the block
// table (or the sequence's contiguous rows); the softmax clears the V rows
// past a sequence in its last block and stores tiles that straddle a
// sequence end row by row.  The MMA and softmax arithmetic is unchanged.
#include <type_traits>

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
    // (+ 128 bytes of static shared memory: the producer's staged rows, ragged/paged gathers)
    static_assert(SMEM_BYTES + 128 <= 227 * 1024, "shared memory budget");
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

// Ragged mode: also the unit's sequence, head and extents.
struct RaggedUnit : Unit {
    int s, h, q_start, kv_start, Nq, Nk;
};

template <bool RAGGED>
using UnitOf = typename std::conditional<RAGGED, RaggedUnit, Unit>::type;

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
    return g;  // the ragged-mode fields stay unset: the dense mode reads the launch's extents
}

// Ragged mode: unit u of the list the schedule pass wrote, entries
// (s, pair, h, q_start) and (q_len, kv_len, kv_start, 0).
__device__ __forceinline__ RaggedUnit ragged_unit(const PrefillParams& p, int u) {
    const int4 a = __ldg(p.units + 2 * u), c = __ldg(p.units + 2 * u + 1);
    RaggedUnit g;
    g.s = a.x;
    g.h = a.z;
    g.bh = a.z;
    g.q_start = a.w;
    g.Nq = c.x;
    g.Nk = c.y;
    g.kv_start = c.z;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        g.q0[t] = (2 * a.y + t) * 128;
        const int rr = g.Nq - g.q0[t];
        g.rows[t] = rr < 0 ? 0 : (rr > 128 ? 128 : rr);
        g.n[t] = tile_blocks(g.q0[t], g.rows[t], g.Nq, g.Nk, p.causal);
    }
    g.J = g.n[0] > g.n[1] ? g.n[0] : g.n[1];
    return g;
}

template <bool RAGGED>
__device__ __forceinline__ UnitOf<RAGGED> unit_at(const PrefillParams& p, int u) {
    if constexpr (RAGGED)
        return ragged_unit(p, u);
    else
        return unit_geometry(p, u);
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

template <int D, bool FP8, bool RAGGED>
__device__ void producer_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                              int n_units) {
    using C = Cfg<D, FP8>;
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    int kv_idx = 0;
    int qcnt[2] = {0, 0};
    int round_ = 0;
    bool ok = true;
    for (int u = next_unit(RAGGED ? n_units : p.n_units, round_); ok && u >= 0; u = next_unit(RAGGED ? n_units : p.n_units, round_)) {
        const UnitOf<RAGGED> g = unit_at<RAGGED>(p, u);
        // The unit's query tiles first, each as soon as the previous unit's
        // last S MMA released its buffer (about when the ring frees the slot
        // for the unit's first K block): Q comes from HBM, as no other unit
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
        for (int j = 0; ok && j < g.J; ++j)
            ok = load_kv<D, FP8>(p, smem, b, abort_flag, kv_idx, j, g.bh, false) &&
                 load_kv<D, FP8>(p, smem, b, abort_flag, kv_idx, j, g.bh, true);
    }
    // Drain: every copy this thread started must land before the CTA exits.
    for (int t = 0; t < 2; ++t)
        if (qcnt[t] > 0) drain_wait(&b.q_full[t], (uint32_t)((qcnt[t] - 1) & 1), p.status);
    for (int idx = kv_idx - C::NST > 0 ? kv_idx - C::NST : 0; idx < kv_idx; ++idx)
        drain_wait(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), p.status);
}

// Ragged mode producer (one warp): the same stream as producer_role -- the
// unit's Q tiles, then K_j, V_j of every KV block -- with
// each 128-key block gathered from 128 / R boxes of R rows: through the block
// table (paged keys) or from the sequence's contiguous rows.  A box past the
// sequence's keys, or naming an out-of-range page, reads the zero fill past
// the end of the key tensor.  The lanes look up the rows of 32 boxes at a
// time (one load latency for all, staged in shared memory); lane 0 alone then
// waits for the slots and issues the copies of those boxes' blocks.  (Lanes
// that meet around every barrier wait -- one lane waiting, the rest at a
// shuffle -- were measured to leave the copies late.)
template <int D>
__device__ void ragged_producer_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                                     int lane, int n_units) {
    using C = Cfg<D, false>;
    __shared__ int s_rows[32];
    if (lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
    }
    const int R = p.rows_per_box;
    const int LPB = 128 / R;  // boxes per block (1..16), a divisor of 32
    const int oob = p.kv_rows;
    const int pshift = p.block_table != nullptr ? __ffs(p.page_size) - 1 : 0;  // page_size is a power of two
    int kv_idx = 0;
    int qcnt[2] = {0, 0};
    int round_ = 0;
    bool ok = true;
    for (int u = next_unit(n_units, round_); ok && u >= 0; u = next_unit(n_units, round_)) {
        const RaggedUnit g = ragged_unit(p, u);
        const int kvh = g.h / p.G;
        const int32_t* bt = p.block_table != nullptr ? p.block_table + (size_t)g.s * p.max_pages : nullptr;
        const int n_boxes = g.J * LPB;
        for (int box0 = 0; ok && box0 < n_boxes; box0 += 32) {
            __syncwarp();  // lane 0 has read the previous batch
            {
                const int key = (box0 + lane) * R;
                int row = oob;
                if (box0 + lane < n_boxes && key < g.Nk) {
                    if (bt == nullptr) {
                        row = g.kv_start + key;
                    } else {
                        const int id = __ldg(bt + (key >> pshift));
                        if (id >= 0 && id < p.num_pages)
                            row = (id << pshift) + (key & (p.page_size - 1));
                        else
                            atomicOr(p.status, 1u << kStatusDeviceData);
                    }
                }
                s_rows[lane] = row;
            }
            __syncwarp();
            if (lane == 0) {
                // the unit's query tiles first (as in producer_role)
                if (box0 == 0) {
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
                            tma_load_3d(smem + C::OFF_Q + t * C::TILE_BYTES + pn * C::PANEL_BYTES, &p.tm_q,
                                        &b.q_full[t], pn * C::PANEL, g.q_start + g.q0[t], g.h);
                        ++qcnt[t];
                    }
                }
                const int j_end = min(g.J, (box0 + 32) / LPB);
                for (int j = box0 / LPB; ok && j < j_end; ++j) {
                    for (int kv = 0; kv < 2; ++kv) {
                        const int slot = kv_idx % C::NST, round = kv_idx / C::NST;
                        if (round > 0 &&
                            !wait_bar(&b.kv_empty[slot], (uint32_t)((round - 1) & 1), abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        bar_arrive_expect_tx(&b.kv_full[slot], C::TILE_BYTES);
                        const CUtensorMap* map = kv ? &p.tm_v : &p.tm_k;
                        uint8_t* dst = smem + C::OFF_KV + slot * C::TILE_BYTES;
                        for (int i = 0; i < LPB; ++i) {
                            const int row = s_rows[j * LPB + i - box0];
#pragma unroll
                            for (int pn = 0; pn < C::NPANEL; ++pn)
                                tma_load_3d(dst + pn * C::PANEL_BYTES + i * R * 128, map, &b.kv_full[slot],
                                            pn * C::PANEL, row, kvh);
                        }
                        ++kv_idx;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
    }
    // Drain: every copy lane 0 started must land before the CTA exits.
    if (lane == 0) {
        for (int t = 0; t < 2; ++t)
            if (qcnt[t] > 0) drain_wait(&b.q_full[t], (uint32_t)((qcnt[t] - 1) & 1), p.status);
        for (int idx = kv_idx - C::NST > 0 ? kv_idx - C::NST : 0; idx < kv_idx; ++idx)
            drain_wait(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), p.status);
    }
    __syncwarp();
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
template <int D, bool FP8, bool RAGGED>
__device__ void mma_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                         uint32_t tmem, int t, int n_units) {
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
    for (int u = next_unit(RAGGED ? n_units : p.n_units, round_); u >= 0; u = next_unit(RAGGED ? n_units : p.n_units, round_)) {
        const UnitOf<RAGGED> g = unit_at<RAGGED>(p, u);
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

// Ragged mode, once per unit: wait for V block iV and zero its row r if r >=
// n_valid (keys past the sequence); warp-collective.  Kept out of line so the
// softmax loop does not hold its registers.
template <int D>
__device__ __noinline__ bool clear_v_tail(uint8_t* smem, const Bars& b, volatile int* abort_flag, unsigned* status,
                                          int iV, int r, int n_valid) {
    using C = Cfg<D, false>;
    const bool ok = __all_sync(0xffffffffu, wait_bar(&b.kv_full[iV % C::NST], (uint32_t)((iV / C::NST) & 1),
                                                     abort_flag, status));
    if (!ok) return false;
    if (r >= n_valid) {
        const uint32_t vrow = smem_u32(smem + C::OFF_KV + (iV % C::NST) * C::TILE_BYTES) + (uint32_t)(r * 128);
#pragma unroll
        for (int pn = 0; pn < C::NPANEL; ++pn)
#pragma unroll
            for (int cb = 0; cb < 128; cb += 16) st_shared_v4(vrow + (uint32_t)(pn * C::PANEL_BYTES + cb), 0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    return true;
}

template <int D, bool FP8, bool RAGGED>
__device__ void softmax_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                             uint32_t tmem, int t, int wq, int lane, int n_units) {
    using C = Cfg<D, FP8>;
    const int r = wq * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::tm_s(t);
    const uint32_t tO = tmem + lane_off + C::tm_o(t);
    const float cs = p.c_scale;
    uint8_t* ost = smem + C::OFF_OST + (t * 4 + wq) * C::OST_WARP_BYTES;
    const uint32_t ost_u = smem_u32(ost);
    uint32_t sblk = 0, units = 0, nstore = 0;
    int round_ = 0, kv_base = 0;
    bool ok = true;

    for (int u = next_unit(RAGGED ? n_units : p.n_units, round_); ok && u >= 0; u = next_unit(RAGGED ? n_units : p.n_units, round_)) {
        const UnitOf<RAGGED> g = unit_at<RAGGED>(p, u);
        const int q0 = g.q0[t], rows = g.rows[t], nt = g.n[t], bh = g.bh;
        const int kvb = kv_base;  // the unit's first K/V stream index
        kv_base += 2 * g.J;
        if (rows <= 0) continue;  // tile lies entirely past Nq
        int Nq_u, Nk_u;  // the unit's sequence
        if constexpr (RAGGED) {
            Nq_u = g.Nq;
            Nk_u = g.Nk;
        } else {
            Nq_u = p.Nq;
            Nk_u = p.Nk;
        }
        const int off = Nk_u - Nq_u;
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
                (kbase + 128 > Nk_u) || (p.causal && (long long)kbase + 127 > (long long)q0 + off);
            if (need_mask) {
                // visible columns of this row: [0, bound), the keys up to
                // min(Nk - 1, limit) (causal) or Nk - 1
                long long last = (long long)Nk_u - 1;
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
            if constexpr (RAGGED) {
                // Keys past the sequence in this block: clear their V rows (a
                // partial last page holds arbitrary bytes, maybe NaN, and
                // 0 * NaN would poison P V).  The tile whose PV reads the
                // block first clears it: tile 0 while it is active, else tile 1.
                if (kbase + 128 > Nk_u && (t == 0 || it >= g.n[0])) {
                    ok = clear_v_tail<D>(smem, b, abort_flag, p.status, kvb + 2 * it + 1, r, Nk_u - kbase);
                    if (!ok) break;
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
        const bool warp_rows = q0 + wq * 32 < Nq_u;        // some row of this warp is inside the sequence
        const bool warp_full = !RAGGED || q0 + wq * 32 + 32 <= Nq_u;  // ragged: all 32 (else direct stores)
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
            if constexpr (!RAGGED) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    st_shared_v4(buf + (uint32_t)(lane * 64 + i * 16), w[4 * i], w[4 * i + 1], w[4 * i + 2],
                                 w[4 * i + 3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (warp_rows) tma_store_3d(&p.tm_o, ost + (nstore & 1u) * 2048u, ch * 32, q0 + wq * 32, bh);
                    tma_store_commit();  // one (possibly empty) group per buffer use keeps the count exact
                }
            } else {
                if (warp_full) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_shared_v4(buf + (uint32_t)(lane * 64 + i * 16), w[4 * i], w[4 * i + 1], w[4 * i + 2],
                                     w[4 * i + 3]);
                    fence_async_smem();
                } else if (r < rows) {  // the warp straddles the sequence end: this row directly
                    uint4* dst =
                        reinterpret_cast<uint4*>(p.o + ((size_t)(g.q_start + row) * p.H + g.h) * D + ch * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
                __syncwarp();
                if (lane == 0) {
                    if (warp_rows && warp_full)
                        tma_store_3d(&p.tm_o, ost + (nstore & 1u) * 2048u, ch * 32, g.q_start + q0 + wq * 32, g.h);
                    tma_store_commit();  // one (possibly empty) group per buffer use keeps the count exact
                }
            }
            ++nstore;
        }
        if (p.lse != nullptr && r < rows) {
            size_t li;
            if constexpr (RAGGED)
                li = (size_t)(g.q_start + row) * p.H + g.h;
            else
                li = (size_t)bh * p.Nq + row;
            p.lse[li] = (l > 0.f) ? (m_use + lg2(l)) * kLn2 : -INFINITY;
        }
    }
    if (lane == 0) tma_store_wait_all();
}

// ---------------------------------------------------------------- kernel

template <int D, bool FP8, bool RAGGED>
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

    if (threadIdx.x == 0) *skip = timeout_recorded(p.status) ? 1 : 0;
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
    // ragged mode: the schedule pass (an earlier kernel of the stream) wrote the unit count
    const int n_units = RAGGED ? __ldg(p.n_listed) : p.n_units;

    if (warp >= 3) {
        // warps 3-6: tile 0, warps 7-10: tile 1; a warp reaches TMEM lanes 32*(warp % 4)..+31
        softmax_role<D, FP8, RAGGED>(p, smem, b, abort_flag, tmem, (warp - 3) >> 2, warp & 3, lane, n_units);
    } else if (warp < 2) {
        if (lane == 0) {
            mma_role<D, FP8, RAGGED>(p, smem, b, abort_flag, tmem, warp, n_units);
            // every issued MMA must finish before tensor memory is released
            tc_commit(&b.done[warp]);
            drain_wait(&b.done[warp], 0, p.status);
        }
        __syncwarp();
    } else {
        if constexpr (RAGGED) {
            ragged_producer_role<D>(p, smem, b, abort_flag, lane, n_units);
        } else {
            if (lane == 0) producer_role<D, FP8, RAGGED>(p, smem, b, abort_flag, n_units);
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

template <int D, bool FP8, bool RAGGED = false>
cudaError_t launch_one(const PrefillParams& p, int grid, cudaStream_t stream) {
    using C = Cfg<D, FP8>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, FP8, RAGGED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prefill_kernel<D, FP8, RAGGED><<<grid, kPrefillThreads, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- ragged schedule pass

constexpr int kRBuckets = 64;

constexpr int kRGroups = 16;
constexpr long long kRGroupBytes = 32ll << 20;
constexpr int kRGroupSeqs = 4096;  // grouping for launches of up to this many sequences
static_assert(kRGroups * kRBuckets == 1024, "one (group, bucket) counter per thread");

// Exclusive scan of one value per thread of a 1024-thread block; `warp_sums`
// holds 32 entries.  Returns the thread's exclusive prefix; *total the sum.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* warp_sums, T* total) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        T z = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const T y = __shfl_up_sync(0xffffffffu, z, o);
            if (lane >= o) z += y;
        }
        warp_sums[lane] = z;  // inclusive
    }
    __syncthreads();
    const T before = (w > 0 ? warp_sums[w - 1] : (T)0) + x - v;
    *total = warp_sums[31];
    __syncthreads();
    return before;
}

// One CTA: every (sequence, query-tile pair) whose first tile has rows,
// bucketed by the KV blocks it streams (longest first; 63 blocks or more
// share the first bucket), each followed by its H heads (heads of one KV
// head adjacent, so units that read the same keys run together).  Offsets or
// lengths out of range are reported in the status word and clamped: a bad
// query range drops the sequence, a bad key range reads no keys.
//
// Sequences are taken in groups -- longest sequences first, a new group
// each time their running K/V bytes cross a multiple of kRGroupBytes -- and
// the list runs group after group, longest first within a group: the units
// running at once then read the K/V of one group, which stays in L2
// (measured on GB300: DRAM reads of a varlen launch of 16 sequences,
// 147 MB of K/V, 879 -> 504 MB; chunks of 8 x 2048 over 6144 cached keys
// 2.04 -> 0.50 GB).  The price is balance: the per-CTA work of the static
// snake order over the list is less even at group boundaries (the varlen
// launch 3% slower, the chunks 2% faster).
__global__ void __launch_bounds__(1024) ragged_schedule_kernel(const RaggedSched sp, int max_pairs) {
    __shared__ int s_bucket[kRGroups * kRBuckets];
    __shared__ unsigned char s_grp[kRGroupSeqs];
    __shared__ int s_isum[32];
    const int t = threadIdx.x;
    s_bucket[t] = 0;  // kRGroups * kRBuckets == 1024 entries
    __syncthreads();
    // extent of sequence s; the report is made once, by its pair-0 group
    auto extent = [&](int s, bool report, int& qs, int& ql, int& kl, int& ks) {
        bool bad = false;
        const int a = __ldg(sp.cu_q + s), e = __ldg(sp.cu_q + s + 1);
        qs = a;
        ql = e - a;
        if (a < 0 || e < a || e > sp.total_q || ql > sp.max_q_len) {
            bad = true;
            qs = 0;
            ql = 0;
        }
        ks = 0;
        if (sp.cu_k != nullptr) {
            const int c = __ldg(sp.cu_k + s), f = __ldg(sp.cu_k + s + 1);
            kl = f - c;
            ks = c;
            if (c < 0 || f < c || f > sp.kv_cap) {
                bad = true;
                kl = 0;
                ks = 0;
            }
        } else {
            kl = __ldg(sp.seq_lens + s);
            if (kl < 0 || kl > sp.kv_cap) {
                bad = true;
                kl = kl < 0 ? 0 : sp.kv_cap;
            }
        }
        if (bad && report) atomicOr(sp.status, 1u << kStatusDeviceData);
    };
    auto blocks = [&](int pair, int ql, int kl) {
        int J = 0;
        for (int tt = 0; tt < 2; ++tt) {
            const int q0 = (2 * pair + tt) * 128, rr = ql - q0;
            const int n = tile_blocks(q0, rr < 0 ? 0 : (rr > 128 ? 128 : rr), ql, kl, sp.causal);
            J = n > J ? n : J;
        }
        return J;
    };
    auto bucket = [](int J) { return J >= kRBuckets - 1 ? 0 : kRBuckets - 1 - J; };
    // group of each sequence (all in group 0 past kRGroupSeqs sequences):
    // the sequences taken longest first (by the KV blocks of their last tile
    // pair, a counting sort over the buckets; ties in any order), cut where
    // the running K/V bytes cross a multiple of kRGroupBytes
    const bool grouped = sp.B <= kRGroupSeqs;
    if (grouped) {
        __shared__ unsigned long long s_bbytes[kRBuckets];
        if (t < kRBuckets) s_bbytes[t] = 0ull;
        __syncthreads();
        auto seq_bucket = [&](int s, long long& bytes) {
            int qs, ql, kl, ks;
            extent(s, false, qs, ql, kl, ks);
            bytes = (long long)kl * sp.kv_bytes_per_key;
            const int last_pair = ql > 0 ? (ql - 1) / 256 : 0;
            return bucket(blocks(last_pair, ql, kl));
        };
        for (int s = t; s < sp.B; s += 1024) {
            long long by;
            const int bk = seq_bucket(s, by);
            atomicAdd(&s_bbytes[bk], (unsigned long long)by);
        }
        __syncthreads();
        if (t == 0) {  // bucket byte totals -> exclusive offsets (64 entries)
            unsigned long long run = 0ull;
            for (int i = 0; i < kRBuckets; ++i) {
                const unsigned long long x = s_bbytes[i];
                s_bbytes[i] = run;
                run += x;
            }
        }
        __syncthreads();
        for (int s = t; s < sp.B; s += 1024) {
            long long by;
            const int bk = seq_bucket(s, by);
            const unsigned long long at = atomicAdd(&s_bbytes[bk], (unsigned long long)by);
            const unsigned long long gidx = at / (unsigned long long)kRGroupBytes;
            s_grp[s] = (unsigned char)(gidx < (unsigned long long)kRGroups ? gidx : kRGroups - 1);
        }
        __syncthreads();
    }
    auto slot = [&](int s, int J) { return (grouped ? (int)s_grp[s] * kRBuckets : 0) + bucket(J); };
    const int n_groups = sp.B * max_pairs;
    for (int gi = t; gi < n_groups; gi += 1024) {
        const int s = gi / max_pairs, pair = gi % max_pairs;
        int qs, ql, kl, ks;
        extent(s, pair == 0, qs, ql, kl, ks);
        if (pair * 256 >= ql) continue;
        atomicAdd(&s_bucket[slot(s, blocks(pair, ql, kl))], sp.H);
    }
    __syncthreads();
    {  // exclusive scan of the (group, bucket) counts
        int total;
        const int excl = block_exclusive_scan<int>(s_bucket[t], s_isum, &total);
        s_bucket[t] = excl;
        if (t == 0) *sp.n_listed = total;
    }
    __syncthreads();
    for (int gi = t; gi < n_groups; gi += 1024) {
        const int s = gi / max_pairs, pair = gi % max_pairs;
        int qs, ql, kl, ks;
        extent(s, false, qs, ql, kl, ks);
        if (pair * 256 >= ql) continue;
        const int pos = atomicAdd(&s_bucket[slot(s, blocks(pair, ql, kl))], sp.H);
        for (int h = 0; h < sp.H; ++h) {
            sp.units[2 * (pos + h)] = make_int4(s, pair, h, qs);
            sp.units[2 * (pos + h) + 1] = make_int4(ql, kl, ks, 0);
        }
    }
}

}  // namespace

int prefill_smem_bytes(int d, bool fp8) {
    if (fp8) return d == 128 ? Cfg<128, true>::SMEM_BYTES : -1;
    if (d == 128) return Cfg<128, false>::SMEM_BYTES;
    if (d == 64) return Cfg<64, false>::SMEM_BYTES;
    return -1;
}

size_t ragged_workspace_bytes(int B, int max_q_len, int H) {
    const size_t pairs = (size_t)((max_q_len + 255) / 256);
    return 256 + (size_t)B * pairs * (size_t)H * 32;
}

cudaError_t launch_ragged_prefill(int d, const RaggedSched& sp, const PrefillParams& p, int grid,
                                  cudaStream_t stream) {
    ragged_schedule_kernel<<<1, 1024, 0, stream>>>(sp, (sp.max_q_len + 255) / 256);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (d == 128) return launch_one<128, false, true>(p, grid, stream);
    if (d == 64) return launch_one<64, false, true>(p, grid, stream);
    return cudaErrorInvalidValue;
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
