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
//   warp 9      TMA producer: Q0, Q1 once, then K_j, V_j into an NST-stage
//               shared-memory ring (mbarrier full/empty pairs).
//   warp 8      MMA issuer (one thread): tcgen05.mma S_t = Q_t K_j^T into
//               tensor memory, and O_t += P_t V_j with P_t read from tensor
//               memory.  Completion is signalled with tcgen05.commit.
//   warps 0-3   softmax for query tile 0 (rows 0..127 of the CTA's 256),
//   warps 4-7   softmax for query tile 1: one thread per row reads its S row
//               from tensor memory, masks, updates (m, l), writes P (bf16 or
//               e4m3) back into tensor memory over S, rescales O when the
//               running max moved by more than kTau (log2 units), and runs
//               the epilogue (O / l -> bf16 -> TMA store, LSE).
//
// Issue order of the MMA thread per KV block j (two query tiles ping-pong so
// each softmax overlaps two GEMMs of the other tile):
//   S0(j), PV1(j-1), S1(j), PV0(j)
// tcgen05 operations complete in issue order, so the commit that signals
// S_t(j) also proves PV_t(j-1) finished: the softmax warpgroup may then
// rescale O_t and overwrite P_t.
//
// Lazy rescaling: the running max used for the exponentials is raised only
// when the new block max exceeds it by more than kTau; O and l share that
// stale max so O / l is unchanged (the merge identity of section 2.2 step 4
// holds for any common reference point), and p stays <= 2^kTau.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr float kTau = 8.0f;             // log2 units; 2^8 = 256 < 448 (e4m3 max)
constexpr float kLn2 = 0.69314718055994530942f;

template <int D, bool FP8>
struct Cfg {
    static constexpr int EB = FP8 ? 1 : 2;            // bytes per input element
    static constexpr int BN = 128;                    // keys per KV block
    static constexpr int PANEL = 128 / EB;            // elements in one 128-byte row panel
    static constexpr int NPANEL = D / PANEL;          // panels per row
    static constexpr int PANEL_BYTES = 128 * 128;     // 128 rows x 128 B
    static constexpr int TILE_BYTES = NPANEL * PANEL_BYTES;
    static constexpr int MMA_K = FP8 ? 32 : 16;       // K per tcgen05.mma (32 bytes)
    static constexpr int S_STEPS = D / MMA_K;
    static constexpr int PV_STEPS = BN / MMA_K;
    static constexpr int NST = (FP8 || D == 64) ? 6 : 4;
    static constexpr int O_PANELS = D / 64;           // bf16 output panels
    static constexpr int O_TILE_BYTES = O_PANELS * PANEL_BYTES;
    static constexpr bool O_IN_Q = !FP8;              // bf16: stage O in the Q tile
    __host__ __device__ static constexpr uint32_t tm_s(int t) { return t ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256u + (t ? (uint32_t)D : 0u); }
    static constexpr uint32_t TM_COLS = 512;
    static constexpr uint32_t P_STEP_COLS = MMA_K * EB / 4;  // TMEM columns per PV step
    static constexpr uint32_t FMT = FP8 ? 0u : 1u;           // e4m3 / bf16
    static constexpr uint32_t ID_S = idesc_make(128, 128, FMT, false, false);
    static constexpr uint32_t ID_PV = idesc_make(128, D, FMT, false, true);
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + 2 * TILE_BYTES;
    static constexpr int OFF_OST = OFF_KV + NST * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_OST + (O_IN_Q ? 0 : 2 * O_TILE_BYTES);
    static constexpr int N_BARS = 1 + 2 * NST + 2 + 2 + 2 + 1;
    static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // request more than half an SM's shared memory so two CTAs never share
    // one SM's tensor memory (each allocates all 512 columns)
    static constexpr int SMEM_BYTES = (SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024);
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(D % PANEL == 0 && D % 64 == 0, "head dim");
};

struct Bars {
    uint64_t* q_full;
    uint64_t* kv_full;
    uint64_t* kv_empty;
    uint64_t* s_full;  // [2]
    uint64_t* p_full;  // [2]
    uint64_t* o_full;  // [2]
    uint64_t* done;
};

// Wait that ignores the abort flag (used only to drain in-flight async work
// before the CTA releases its shared and tensor memory); bounded in time.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned* status) {
    const unsigned long long t0 = globaltimer();
    while (!bar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(status, 1u << kStatusTimeout);
            return;
        }
    }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// AND of `pred` over the `nthreads` threads of named barrier `id` (all of them
// must arrive); gives every thread of a warpgroup the same decision.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "bar.red.and.pred pout, %2, %3, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

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

template <int D, bool FP8>
__device__ void producer_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                              int bh, const int (&q0)[2], const int (&n)[2]) {
    using C = Cfg<D, FP8>;
    const int J = n[0] > n[1] ? n[0] : n[1];
    if (J == 0) return;
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    const uint32_t qbytes = (n[0] > 0 ? C::TILE_BYTES : 0) + (n[1] > 0 ? C::TILE_BYTES : 0);
    bar_arrive_expect_tx(b.q_full, qbytes);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (n[t] == 0) continue;
#pragma unroll
        for (int pn = 0; pn < C::NPANEL; ++pn)
            tma_load_3d(smem + C::OFF_Q + t * C::TILE_BYTES + pn * C::PANEL_BYTES, &p.tm_q, b.q_full,
                        pn * C::PANEL, q0[t], bh);
    }
    int issued = 0;
    for (int idx = 0; idx < 2 * J; ++idx) {
        const int j = idx >> 1;
        const int slot = idx % C::NST;
        const int round = idx / C::NST;
        if (round > 0 && !wait_bar(&b.kv_empty[slot], (round - 1) & 1, abort_flag, p.status)) break;
        bar_arrive_expect_tx(&b.kv_full[slot], C::TILE_BYTES);
        const CUtensorMap* map = (idx & 1) ? &p.tm_v : &p.tm_k;
        uint8_t* dst = smem + C::OFF_KV + slot * C::TILE_BYTES;
#pragma unroll
        for (int pn = 0; pn < C::NPANEL; ++pn)
            tma_load_3d(dst + pn * C::PANEL_BYTES, map, &b.kv_full[slot], pn * C::PANEL, j * 128, bh);
        issued = idx + 1;
    }
    // Drain: every copy this thread started must land before the CTA exits.
    drain_wait(b.q_full, 0, p.status);
    for (int idx = issued - C::NST > 0 ? issued - C::NST : 0; idx < issued; ++idx)
        drain_wait(&b.kv_full[idx % C::NST], (idx / C::NST) & 1, p.status);
}

template <int D, bool FP8>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
    using C = Cfg<D, FP8>;
#pragma unroll
    for (int k = 0; k < C::S_STEPS; ++k) {
        const uint32_t off = (uint32_t)((k >> 2) * C::PANEL_BYTES + (k & 3) * 32);
        const uint64_t a = sdesc_sw128(q_smem + off, 16, 1024);
        const uint64_t bd = sdesc_sw128(k_smem + off, 16, 1024);
        if (FP8)
            mma_f8_ss(d_tmem, a, bd, C::ID_S, k > 0 ? 1u : 0u);
        else
            mma_f16_ss(d_tmem, a, bd, C::ID_S, k > 0 ? 1u : 0u);
    }
}

template <int D, bool FP8>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem, bool accumulate) {
    using C = Cfg<D, FP8>;
#pragma unroll
    for (int s = 0; s < C::PV_STEPS; ++s) {
        const uint64_t bd = sdesc_sw128(v_smem + (uint32_t)(s * C::MMA_K * 128), C::PANEL_BYTES, 1024);
        const uint32_t acc = (accumulate || s > 0) ? 1u : 0u;
        if (FP8)
            mma_f8_ts(o_tmem, p_tmem + s * C::P_STEP_COLS, bd, C::ID_PV, acc);
        else
            mma_f16_ts(o_tmem, p_tmem + s * C::P_STEP_COLS, bd, C::ID_PV, acc);
    }
}

template <int D, bool FP8>
__device__ void mma_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                         uint32_t tmem, const int (&n)[2]) {
    using C = Cfg<D, FP8>;
    const int J = n[0] > n[1] ? n[0] : n[1];
    if (J == 0) return;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t q_s[2] = {sbase + C::OFF_Q, sbase + C::OFF_Q + C::TILE_BYTES};
    auto kv_smem = [&](int idx) { return sbase + C::OFF_KV + (uint32_t)((idx % C::NST) * C::TILE_BYTES); };
    auto kv_par = [&](int idx) { return (uint32_t)((idx / C::NST) & 1); };

    if (!wait_bar(b.q_full, 0, abort_flag, p.status)) return;
    tc_fence_after();
    for (int j = 0; j <= J; ++j) {
        const int iK = 2 * j, iV = 2 * j + 1;
        if (j < J) {
            if (!wait_bar(&b.kv_full[iK % C::NST], kv_par(iK), abort_flag, p.status)) return;
            tc_fence_after();
            if (j < n[0]) {
                issue_s<D, FP8>(tmem + C::tm_s(0), q_s[0], kv_smem(iK));
                tc_commit(&b.s_full[0]);
            }
        }
        // PV for tile 1 of the previous block
        if (j > 0 && j - 1 < n[1]) {
            const int iVp = 2 * (j - 1) + 1;
            if (!wait_bar(&b.kv_full[iVp % C::NST], kv_par(iVp), abort_flag, p.status)) return;
            if (!wait_bar(&b.p_full[1], (uint32_t)((j - 1) & 1), abort_flag, p.status)) return;
            tc_fence_after();
            issue_pv<D, FP8>(tmem + C::tm_o(1), tmem + C::tm_s(1), kv_smem(iVp), j - 1 > 0);
            tc_commit(&b.kv_empty[iVp % C::NST]);
            if (j - 1 == n[1] - 1) tc_commit(&b.o_full[1]);
        }
        if (j == J) break;
        if (j < n[1]) {
            issue_s<D, FP8>(tmem + C::tm_s(1), q_s[1], kv_smem(iK));
            tc_commit(&b.s_full[1]);
        }
        tc_commit(&b.kv_empty[iK % C::NST]);
        if (j < n[0]) {
            if (!wait_bar(&b.kv_full[iV % C::NST], kv_par(iV), abort_flag, p.status)) return;
            if (!wait_bar(&b.p_full[0], (uint32_t)(j & 1), abort_flag, p.status)) return;
            tc_fence_after();
            issue_pv<D, FP8>(tmem + C::tm_o(0), tmem + C::tm_s(0), kv_smem(iV), j > 0);
            if (j == n[0] - 1) tc_commit(&b.o_full[0]);
            if (!(j < n[1])) tc_commit(&b.kv_empty[iV % C::NST]);
        }
    }
}

template <int D, bool FP8>
__device__ void softmax_role(const PrefillParams& p, uint8_t* smem, const Bars& b, volatile int* abort_flag,
                             uint32_t tmem, int t, int wq, int lane, int bh, int q0, int rows, int n_t) {
    using C = Cfg<D, FP8>;
    if (rows <= 0) return;  // tile lies entirely past Nq
    const int r = wq * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::tm_s(t);
    const uint32_t tO = tmem + lane_off + C::tm_o(t);
    const int row = q0 + r;
    const int off = p.Nk - p.Nq;
    const long long limit = (long long)row + off;  // last visible key (causal)
    const float cs = p.c_scale;

    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < n_t; ++it) {
        // every lane of the warp takes the same branch (tcgen05.ld is warp-collective)
        ok = __all_sync(0xffffffffu, wait_bar(&b.s_full[t], (uint32_t)(it & 1), abort_flag, p.status));
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
        const bool need_mask = (kbase + 128 > p.Nk) || (p.causal && (long long)kbase + 127 > (long long)q0 + off);
        if (need_mask) {
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                const int key = kbase + c;
                if (key >= p.Nk || (p.causal && (long long)key > limit)) s[c] = __float_as_uint(-INFINITY);
            }
        }
        float mx = __uint_as_float(s[0]);
#pragma unroll
        for (int c = 1; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
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
        float rowsum = 0.f;
        if (FP8) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float p0 = ex2(fmaf(__uint_as_float(s[4 * i + 0]), cs, -m_use));
                const float p1 = ex2(fmaf(__uint_as_float(s[4 * i + 1]), cs, -m_use));
                const float p2 = ex2(fmaf(__uint_as_float(s[4 * i + 2]), cs, -m_use));
                const float p3 = ex2(fmaf(__uint_as_float(s[4 * i + 3]), cs, -m_use));
                rowsum += (p0 + p1) + (p2 + p3);
                w[i] = pack_e4m3x4(p0, p1, p2, p3);
            }
            tmem_st32(tS, w);
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float p0 = ex2(fmaf(__uint_as_float(s[64 * h + 2 * i + 0]), cs, -m_use));
                    const float p1 = ex2(fmaf(__uint_as_float(s[64 * h + 2 * i + 1]), cs, -m_use));
                    rowsum += p0 + p1;
                    w[i] = pack_bf16(p0, p1);
                }
                tmem_st32(tS + 32 * h, w);
            }
        }
        l += rowsum;
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

    // ---- epilogue: O / l -> bf16 -> shared (128B-swizzled) -> TMA store; LSE
    if (ok && n_t > 0) {
        ok = __all_sync(0xffffffffu, wait_bar(&b.o_full[t], 0, abort_flag, p.status));
        tc_fence_after();
    }
    // one decision for the whole warpgroup before its named barriers
    ok = named_bar_and(1 + t, 128, ok);
    if (!ok) return;
    const float m_use = (m == -INFINITY) ? 0.f : m;
    const float inv = (l > 0.f) ? p.o_scale / l : 0.f;
    uint8_t* stage = C::O_IN_Q ? smem + C::OFF_Q + t * C::TILE_BYTES : smem + C::OFF_OST + t * C::O_TILE_BYTES;
    const uint32_t stage_u = smem_u32(stage);
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        if (n_t > 0) {
            tmem_ld32(tO + 32 * ch, o);
            tmem_ld_wait();
            reg_after_wait<32>(o);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        const uint32_t panel_base = stage_u + (uint32_t)((ch >> 1) * C::PANEL_BYTES + r * 128);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t chunk = (uint32_t)((ch & 1) * 4 + i);
            st_shared_v4(panel_base + ((chunk ^ (uint32_t)(r & 7)) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2],
                         w[4 * i + 3]);
        }
    }
    fence_async_smem();
    named_bar_sync(1 + t, 128);
    if (r == 0) {
#pragma unroll
        for (int pn = 0; pn < C::O_PANELS; ++pn)
            tma_store_3d(&p.tm_o, stage + pn * C::PANEL_BYTES, pn * 64, q0, bh);
        tma_store_commit();
        tma_store_wait_all();
    }
    if (p.lse != nullptr && r < rows)
        p.lse[(size_t)bh * p.Nq + row] = (l > 0.f) ? (m_use + lg2(l)) * kLn2 : -INFINITY;
}

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
    b.kv_full = bars + 1;
    b.kv_empty = bars + 1 + C::NST;
    b.s_full = bars + 1 + 2 * C::NST;
    b.p_full = b.s_full + 2;
    b.o_full = b.p_full + 2;
    b.done = b.o_full + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

    if (threadIdx.x == 0) *skip = (*(volatile unsigned*)p.status != 0u) ? 1 : 0;
    __syncthreads();
    if (*skip) return;  // an earlier launch gave up: leave the device quiet

    // work unit: heaviest (last) query-tile pairs first, all heads of a pair adjacent
    const int pair = p.n_pairs - 1 - (int)(blockIdx.x / (unsigned)p.BH);
    const int bh = (int)(blockIdx.x % (unsigned)p.BH);
    int q0[2], rows[2], n[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        q0[t] = (2 * pair + t) * 128;
        const int rr = p.Nq - q0[t];
        rows[t] = rr < 0 ? 0 : (rr > 128 ? 128 : rr);
        n[t] = tile_blocks(q0[t], rows[t], p.Nq, p.Nk, p.causal);
    }

    if (threadIdx.x == 0) {
        bar_init(b.q_full, 1);
        for (int s = 0; s < C::NST; ++s) {
            bar_init(&b.kv_full[s], 1);
            bar_init(&b.kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            bar_init(&b.s_full[t], 1);
            bar_init(&b.p_full[t], 128);
            bar_init(&b.o_full[t], 1);
        }
        bar_init(b.done, 1);
        *abort_flag = 0;
        bar_init_fence();
    }
    if (warp == 8) {
        tmem_alloc(tmem_holder, C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp < 8) {
        const int t = warp >> 2;
        softmax_role<D, FP8>(p, smem, b, abort_flag, tmem, t, warp & 3, lane, bh, q0[t], rows[t], n[t]);
    } else if (warp == 8) {
        if (lane == 0) {
            mma_role<D, FP8>(p, smem, b, abort_flag, tmem, n);
            // every issued MMA must finish before tensor memory is released
            tc_commit(b.done);
            drain_wait(b.done, 0, p.status);
        }
        __syncwarp();
    } else {
        if (lane == 0) producer_role<D, FP8>(p, smem, b, abort_flag, bh, q0, n);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

template <int D, bool FP8>
cudaError_t launch_one(const PrefillParams& p, int grid, cudaStream_t stream) {
    using C = Cfg<D, FP8>;
    static_assert(C::SMEM_BYTES > 0, "");
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
