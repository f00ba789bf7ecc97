// backward.cu -- gradients of exact attention (dQ, dK, dV) by recomputation.
//
// The forward pass keeps only the row statistics (here the LSE); the
// backward pass recomputes the probabilities on chip from Q, K and those
// statistics instead of reading a stored N x N matrix ("Capstone: CUDA
// Softmax 与 Attention 算子", section 6.1, the pitfalls table, and section 7.3,
// question 1).  The gradient of O = softmax(scale Q K^T) V for an upstream
// gradient dO is, per query row i and key j:
//   P_ij = 2^(scale log2(e) q_i.k_j - lse_i log2(e)),   D_i = dO_i . O_i
//   dV_j += P_ij dO_i,   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i)
//   dQ_i += scale dS_ij k_j,   dK_j += scale dS_ij q_i
//
// Three kernels:
//   bwd_prep    D = rowsum(dO * O) and lse2 = lse log2(e) (+inf for rows
//               with no visible key, so their P is 0), both padded to whole
//               128-row blocks; zeroes the fp32 dQ accumulator.
//   bwd_main    (d = 64; d = 128 runs bwd_pipe, described further down: the
//               same products on 64-query blocks, pipelined across blocks,
//               one persistent CTA per SM)
//               one CTA per (batch*head, 128-key block j), K_j and V_j
//               resident in shared memory, looping over the query blocks i
//               that see any of its keys (all blocks, or from the diagonal on
//               under the causal mask):
//                 warp 0    TMA: K_j, V_j once; Q_i and dO_i double-buffered
//                 warp 1    MMA issuer (one thread):
//                             S^T = K_j Q_i^T, dP^T = V_j dO_i^T  (TMEM, keys on lanes)
//                             dV += P^T dO_i, dK += dS^T Q_i       (A = P^T / dS^T from TMEM)
//                             dQ_i = dS K_j                       (A = dS from shared memory)
//                 warps 2-5 one thread per key: P^T and dS^T from S^T, dP^T, lse2, D
//                           (the block's lse2 and D staged in shared memory, one entry
//                           per thread; masked pairs: 0); P^T, dS^T back to TMEM as bf16 and dS to
//                           shared memory in the layout the dQ product reads;
//                           at the end dK (times scale) and dV -> bf16 -> global
//                 warps 6-9 one thread per query: dQ_i from TMEM to registers (TMEM
//                           released at once), staged in the block's own Q / dO slot
//                           (free once the products reading it are done) and added
//                           into the fp32 accumulator by bulk tensor reductions
//   bwd_dq      dQ = scale * accumulator -> bf16.
//
// Tensor memory: columns 0-127 S^T, then P^T over it, then dQ_i; 128-255
// dP^T, then dS^T over it; 256.. dV (d columns); 256 + d.. dK (d columns).
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace attn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BCfg {
    static constexpr int NPANEL = D / 64;
    static constexpr int PANEL_BYTES = 128 * 128;
    static constexpr int TILE_BYTES = NPANEL * PANEL_BYTES;  // 128 rows x d bf16
    static constexpr int DS_BYTES = 2 * PANEL_BYTES;         // 128 keys x 128 queries bf16
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE_BYTES;
    static constexpr int OFF_Q = OFF_V + TILE_BYTES;        // [2]
    static constexpr int OFF_DO = OFF_Q + 2 * TILE_BYTES;   // [2]
    static constexpr int OFF_DS = OFF_DO + 2 * TILE_BYTES;
    static constexpr int OFF_LD = OFF_DS + DS_BYTES;        // lse2[128], D[128] of the current query block
    static constexpr int OFF_BAR = OFF_LD + 2 * 128 * 4;
    static constexpr int N_BARS = 12;
    static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = (SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024);
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(2 * (D / 32) * 4096 <= TILE_BYTES, "two warps' dQ staging fits one Q or dO slot");
    // dQ = dS K: A = dS (MN-major: queries contiguous), B = K_j (MN-major: dims contiguous)
    static constexpr uint32_t ID_DQ = idesc_make(128, D, 1u, true, true);
};

struct BBars {
    uint64_t* kv_full;
    uint64_t* qd_full;   // [2]
    uint64_t* qd_empty;  // [2], the products reading Q_i / dO_i done (1) and dQ_i staged out of the slot (4)
    uint64_t* s_full;    // S^T and dP^T computed
    uint64_t* ds_ready;  // 128 arrivals: P^T, dS^T in TMEM, dS in shared memory
    uint64_t* dq_full;   // dQ_i computed (also: dS in shared memory consumed)
    uint64_t* dq_empty;  // 128 arrivals: dQ_i read out of TMEM
    uint64_t* done;      // all products finished (dK, dV final)
    uint64_t* ld_full;   // 128 arrivals: lse2 / D of the block staged in shared memory
    uint64_t* ld_free;   // 128 arrivals: every dS thread has finished reading them
};

// Query blocks a key block j sees: [i0, n_qb).  Under the causal mask query
// q sees key k iff k <= q + (Nk - Nq), so block i is needed iff its last
// query reaches the block's first key.
__device__ __forceinline__ int first_qblock(const BwdParams& p, int j) {
    if (!p.causal) return 0;
    const long long need = (long long)j * 128 - (p.Nk - p.Nq) - 127;  // smallest useful last-query index
    if (need <= 0) return 0;
    return (int)((need + 127) / 128);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_global_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ---------------------------------------------------------------- prep / dq kernels

// One warp per padded query row: D and lse2 (padding rows: D = 0, lse2 =
// +inf), and the row's dQ accumulator zeroed.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdParams p) {
    constexpr int PER = D / 32;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (long long)p.BH * p.nq_pad) return;
    const int bh = (int)(gw / p.nq_pad), i = (int)(gw % p.nq_pad);
    float dsum = 0.f, l2 = INFINITY;
    if (i < p.Nq) {
        const size_t row = ((size_t)bh * p.Nq + i) * D + lane * PER;
        const uint16_t* o = p.o + row;
        const uint16_t* g = p.dout + row;
#pragma unroll
        for (int c = 0; c < PER; c += 2) {
            const uint32_t ow = *reinterpret_cast<const uint32_t*>(o + c);
            const uint32_t gwd = *reinterpret_cast<const uint32_t*>(g + c);
            dsum = fmaf(bf16lo_to_f32(ow), bf16lo_to_f32(gwd), dsum);
            dsum = fmaf(bf16hi_to_f32(ow), bf16hi_to_f32(gwd), dsum);
        }
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, s);
        const float lse = p.lse[(size_t)bh * p.Nq + i];
        l2 = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
    }
    if (lane == 0) {
        p.dvec[gw] = dsum;
        p.lse2[gw] = l2;
    }
    float* acc = p.dq_acc + (size_t)gw * D + lane * PER;
#pragma unroll
    for (int c = 0; c < PER; ++c) acc[c] = 0.f;
}

template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const BwdParams p) {
    constexpr int PER = D / 32;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (long long)p.BH * p.Nq) return;
    const int bh = (int)(gw / p.Nq), i = (int)(gw % p.Nq);
    const float* acc = p.dq_acc + ((size_t)bh * p.nq_pad + i) * D + lane * PER;
    uint16_t* dst = p.dq + (size_t)gw * D + lane * PER;
#pragma unroll
    for (int c = 0; c < PER; c += 2) *reinterpret_cast<uint32_t*>(dst + c) = pack_bf16(acc[c] * p.scale, acc[c + 1] * p.scale);
}

// ---------------------------------------------------------------- main kernel roles

template <int D>
__device__ void bwd_producer(const BwdParams& p, uint8_t* smem, const BBars& b, volatile int* abort_flag, int bh,
                             int j, int i0, int nqb) {
    using C = BCfg<D>;
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    tma_prefetch_map(&p.tm_do);
    bar_arrive_expect_tx(b.kv_full, 2 * C::TILE_BYTES);
#pragma unroll
    for (int pn = 0; pn < C::NPANEL; ++pn) {
        tma_load_3d(smem + C::OFF_K + pn * C::PANEL_BYTES, &p.tm_k, b.kv_full, pn * 64, j * 128, bh);
        tma_load_3d(smem + C::OFF_V + pn * C::PANEL_BYTES, &p.tm_v, b.kv_full, pn * 64, j * 128, bh);
    }
    int issued = 0;
    for (int it = 0; it < nqb; ++it) {
        const int s = it & 1;
        if (it >= 2 && !wait_bar(&b.qd_empty[s], (uint32_t)(((it >> 1) - 1) & 1), abort_flag, p.status)) break;
        const int i = i0 + it;
        bar_arrive_expect_tx(&b.qd_full[s], 2 * C::TILE_BYTES);
#pragma unroll
        for (int pn = 0; pn < C::NPANEL; ++pn) {
            tma_load_3d(smem + C::OFF_Q + s * C::TILE_BYTES + pn * C::PANEL_BYTES, &p.tm_q, &b.qd_full[s], pn * 64,
                        i * 128, bh);
            tma_load_3d(smem + C::OFF_DO + s * C::TILE_BYTES + pn * C::PANEL_BYTES, &p.tm_do, &b.qd_full[s], pn * 64,
                        i * 128, bh);
        }
        ++issued;
    }
    // every copy started here lands before the CTA exits
    drain_wait(b.kv_full, 0, p.status);
    for (int it = issued - 2 > 0 ? issued - 2 : 0; it < issued; ++it)
        drain_wait(&b.qd_full[it & 1], (uint32_t)((it >> 1) & 1), p.status);
}

template <int D>
__device__ void bwd_mma(const BwdParams& p, uint8_t* smem, const BBars& b, volatile int* abort_flag, uint32_t tmem,
                        int nqb) {
    using C = BCfg<D>;
    const uint32_t sb = smem_u32(smem);
    // K-major views (S^T = K Q^T, dP^T = V dO^T) and MN-major views (B of dV, dK, dQ)
    const uint64_t k_kmaj = sdesc_sw128(sb + C::OFF_K, 16, 1024);
    const uint64_t v_kmaj = sdesc_sw128(sb + C::OFF_V, 16, 1024);
    const uint64_t k_mn = sdesc_sw128(sb + C::OFF_K, C::PANEL_BYTES, 1024);
    const uint64_t ds_mn = sdesc_sw128(sb + C::OFF_DS, C::PANEL_BYTES, 1024);
    if (!wait_bar(b.kv_full, 0, abort_flag, p.status)) return;
    for (int it = 0; it < nqb; ++it) {
        const int s = it & 1;
        const uint32_t q_addr = sb + C::OFF_Q + s * C::TILE_BYTES, do_addr = sb + C::OFF_DO + s * C::TILE_BYTES;
        if (!wait_bar(&b.qd_full[s], (uint32_t)((it >> 1) & 1), abort_flag, p.status)) return;
        // the previous dQ_i has left TMEM (its columns are where S^T goes)
        if (it > 0 && !wait_bar(b.dq_empty, (uint32_t)((it - 1) & 1), abort_flag, p.status)) return;
        tc_fence_after();
        issue_s<D, false>(tmem + C::TM_S, k_kmaj, sdesc_sw128(q_addr, 16, 1024));
        issue_s<D, false>(tmem + C::TM_DP, v_kmaj, sdesc_sw128(do_addr, 16, 1024));
        tc_commit(b.s_full);
        if (!wait_bar(b.ds_ready, (uint32_t)(it & 1), abort_flag, p.status)) return;
        tc_fence_after();
        issue_pv<D, false>(tmem + C::TM_DV, tmem + C::TM_S, sdesc_sw128(do_addr, C::PANEL_BYTES, 1024), it > 0);
        issue_pv<D, false>(tmem + C::TM_DK, tmem + C::TM_DP, sdesc_sw128(q_addr, C::PANEL_BYTES, 1024), it > 0);
        tc_commit(&b.qd_empty[s]);
        // dQ_i = dS K_j: 8 steps of 16 keys, both operands advance 16 rows (2 KB)
        mma4_ss<128, 256, 384, 128, 256, 384, false>(tmem + C::TM_S, ds_mn, k_mn, C::ID_DQ, 0u);
        mma4_ss<128, 256, 384, 128, 256, 384, false>(tmem + C::TM_S, ds_mn + 512, k_mn + 512, C::ID_DQ, 1u);
        tc_commit(b.dq_full);
    }
}

// One thread per key row (TMEM lane): P^T, dS^T for each query block, then
// the dK, dV epilogue.
template <int D>
__device__ void bwd_ds_role(const BwdParams& p, uint8_t* smem, const BBars& b, volatile int* abort_flag,
                            uint32_t tmem, int bh, int j, int i0, int nqb, int wq, int lane) {
    using C = BCfg<D>;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S, tP = tmem + lane_off + C::TM_DP;
    const int key = j * 128 + row;
    const bool key_ok = key < p.Nk;
    const int off = p.Nk - p.Nq;
    const float cs = p.c_scale;
    const uint32_t ds_row = smem_u32(smem + C::OFF_DS) + (uint32_t)(row * 128);
    float* lds = reinterpret_cast<float*>(smem + C::OFF_LD);  // [0, 128): -lse2, [128, 256): -D
    // this thread's lse2 / D entry of the next query block, loaded one block ahead
    const float* l2g = p.lse2 + (size_t)bh * p.nq_pad + (size_t)i0 * 128 + row;
    const float* dvg = p.dvec + (size_t)bh * p.nq_pad + (size_t)i0 * 128 + row;
    float nx_l = nqb > 0 ? l2g[0] : 0.f, nx_d = nqb > 0 ? dvg[0] : 0.f;
    bool ok = true;
    for (int it = 0; ok && it < nqb; ++it) {
        const int i = i0 + it;
        // stage the block's lse2 and D once every thread is done with the
        // previous block's, then start loading the following block's
        const float my_l = nx_l, my_d = nx_d;
        if (it + 1 < nqb) {
            nx_l = l2g[(size_t)(it + 1) * 128];
            nx_d = dvg[(size_t)(it + 1) * 128];
        }
        if (it > 0) {
            ok = __all_sync(0xffffffffu, wait_bar(b.ld_free, (uint32_t)((it - 1) & 1), abort_flag, p.status));
            if (!ok) break;
        }
        lds[row] = -my_l;  // stored negated: the score step is one fma, the dS step one add
        lds[128 + row] = -my_d;
        bar_arrive(b.ld_full);
        ok = __all_sync(0xffffffffu, wait_bar(b.ld_full, (uint32_t)(it & 1), abort_flag, p.status));
        if (!ok) break;
        ok = __all_sync(0xffffffffu, wait_bar(b.s_full, (uint32_t)(it & 1), abort_flag, p.status));
        if (!ok) break;
        // dS in shared memory is free once the previous block's dQ product read it
        if (it > 0) {
            ok = __all_sync(0xffffffffu, wait_bar(b.dq_full, (uint32_t)((it - 1) & 1), abort_flag, p.status));
            if (!ok) break;
        }
        tc_fence_after();
        // Queries of this block before `vis_from` do not see this key (causal
        // mask); the whole warp takes the mask-free path when none of its keys
        // needs it.  Scores, shifts and products run as packed pairs.
        const int vis_from = key_ok ? (p.causal ? key - off - i * 128 : 0) : 128;
        const bool all_visible = __all_sync(0xffffffffu, vis_from <= 0);
        const float* nl = lds;        // -lse2 of the block's queries
        const float* nd = lds + 128;  // -D
        const uint64_t cs2 = f2_pack(cs, cs);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {  // 32 queries per chunk
            uint32_t sv[32], dp[32];
            tmem_ld32(tS + 32 * c, sv);
            tmem_ld32(tP + 32 * c, dp);
            tmem_ld_wait();
            reg_after_wait<32>(sv);
            reg_after_wait<32>(dp);
            uint32_t pw[16], dw[16];
#pragma unroll
            for (int t4 = 0; t4 < 8; ++t4) {
                const float4 L = *reinterpret_cast<const float4*>(nl + 32 * c + 4 * t4);
                const float4 Dn = *reinterpret_cast<const float4*>(nd + 32 * c + 4 * t4);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = 4 * t4 + 2 * h;
                    const uint64_t x = f2_fma(f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1])), cs2,
                                              h ? f2_pack(L.z, L.w) : f2_pack(L.x, L.y));
                    float p0, p1;
                    f2_unpack(x, p0, p1);
                    p0 = ex2(p0);
                    p1 = ex2(p1);
                    if (!all_visible) {
                        const int tq = 32 * c + t;  // query index within the block
                        p0 = tq >= vis_from ? p0 : 0.f;
                        p1 = tq + 1 >= vis_from ? p1 : 0.f;
                    }
                    const uint64_t pp = f2_pack(p0, p1);
                    const uint64_t diff = f2_add(f2_pack(__uint_as_float(dp[t]), __uint_as_float(dp[t + 1])),
                                                 h ? f2_pack(Dn.z, Dn.w) : f2_pack(Dn.x, Dn.y));
                    float d0, d1;
                    f2_unpack(f2_mul(pp, diff), d0, d1);
                    pw[2 * t4 + h] = pack_bf16(p0, p1);
                    dw[2 * t4 + h] = pack_bf16(d0, d1);
                }
            }
            tmem_st16(tS + 16 * c, pw);
            tmem_st16(tP + 16 * c, dw);
            // dS row `row`, queries 32c..32c+31: panel c / 2, 16-byte chunks
            // (c % 2) * 4 .. +3 of the row, 128-byte swizzle (chunk ^ row % 8)
            const uint32_t prow = ds_row + (uint32_t)((c >> 1) * C::PANEL_BYTES);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t chunk = (uint32_t)((c & 1) * 4 + k) ^ (uint32_t)(row & 7);
                st_shared_v4(prow + chunk * 16u, dw[4 * k], dw[4 * k + 1], dw[4 * k + 2], dw[4 * k + 3]);
            }
        }
        tmem_st_wait();
        fence_async_smem();
        tc_fence_before();
        bar_arrive(b.ds_ready);
        bar_arrive(b.ld_free);
    }
    if (!ok) return;
    // ---- epilogue: dV and scale * dK rows of this key block -> bf16
    if (nqb > 0) {
        ok = __all_sync(0xffffffffu, wait_bar(b.done, 0, abort_flag, p.status));
        if (!ok) return;
        tc_fence_after();
    }
    uint16_t* dvr = p.dv + ((size_t)bh * p.Nk + key) * D;
    uint16_t* dkr = p.dk + ((size_t)bh * p.Nk + key) * D;
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t a[32], g[32];
        if (nqb > 0) {
            tmem_ld32(tmem + lane_off + C::TM_DV + 32 * ch, a);
            tmem_ld32(tmem + lane_off + C::TM_DK + 32 * ch, g);
            tmem_ld_wait();
            reg_after_wait<32>(a);
            reg_after_wait<32>(g);
        } else {  // no query sees this block: zero gradients
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = g[e] = 0u;
        }
        if (key_ok) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
                st_global_v4(dvr + 32 * ch + e, pack_bf16(__uint_as_float(a[e]), __uint_as_float(a[e + 1])),
                             pack_bf16(__uint_as_float(a[e + 2]), __uint_as_float(a[e + 3])),
                             pack_bf16(__uint_as_float(a[e + 4]), __uint_as_float(a[e + 5])),
                             pack_bf16(__uint_as_float(a[e + 6]), __uint_as_float(a[e + 7])));
                const float sc = p.scale;
                st_global_v4(dkr + 32 * ch + e,
                             pack_bf16(__uint_as_float(g[e]) * sc, __uint_as_float(g[e + 1]) * sc),
                             pack_bf16(__uint_as_float(g[e + 2]) * sc, __uint_as_float(g[e + 3]) * sc),
                             pack_bf16(__uint_as_float(g[e + 4]) * sc, __uint_as_float(g[e + 5]) * sc),
                             pack_bf16(__uint_as_float(g[e + 6]) * sc, __uint_as_float(g[e + 7]) * sc));
            }
        }
    }
}

// One thread per query row of the block (TMEM lane): dQ_i added into the
// accumulator (padded rows, so every row of a block exists).
template <int D>
__device__ void bwd_dq_role(const BwdParams& p, uint8_t* smem, const BBars& b, volatile int* abort_flag,
                            uint32_t tmem, int bh, int i0, int nqb, int wq, int lane) {
    using C = BCfg<D>;
    const uint32_t tQ = tmem + ((uint32_t)(wq * 32) << 16) + C::TM_S;
    if (lane == 0) tma_prefetch_map(&p.tm_dq);
    // this warp's staging area: 32 rows x d fp32, in the Q slot (warps 0, 1) or
    // the dO slot (warps 2, 3) of the block's buffer pair
    const int stage_off = (wq < 2 ? C::OFF_Q : C::OFF_DO) + (wq & 1) * (D / 32) * 4096;
    for (int it = 0; it < nqb; ++it) {
        const int s = it & 1;
        const bool okw = __all_sync(0xffffffffu, wait_bar(b.dq_full, (uint32_t)(it & 1), abort_flag, p.status));
        if (!okw) break;
        tc_fence_after();
        // the whole row into registers first: TMEM is released at once
        uint32_t v[D];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(tQ + 32 * ch, v + 32 * ch);
        tmem_ld_wait();
        reg_after_wait<D>(v);
        tc_fence_before();
        bar_arrive(b.dq_empty);
        // Stage the warp's 32 rows in the block's Q / dO slot (free: the products
        // that read it completed before dQ_i) as D / 32 boxes of 32 rows x 32 fp32
        // (128 B rows, 128-byte swizzle: 16-byte chunk k of row r at k ^ (r % 8)),
        // then let the bulk-copy engine add them into the accumulator.
        uint8_t* stage_p = smem + stage_off + s * C::TILE_BYTES;
        const uint32_t stage = smem_u32(stage_p);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
            const uint32_t rowp = stage + (uint32_t)(ch * 4096 + lane * 128);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                st_shared_v4(rowp + (((uint32_t)k ^ (uint32_t)(lane & 7)) << 4), v[32 * ch + 4 * k],
                             v[32 * ch + 4 * k + 1], v[32 * ch + 4 * k + 2], v[32 * ch + 4 * k + 3]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            const int row0 = (i0 + it) * 128 + wq * 32;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch)
                tma_reduce_add_3d(&p.tm_dq, stage_p + ch * 4096, ch * 32, row0, bh);
            tma_store_commit();
            tma_wait_read_all();  // the slot may be refilled once the engine has read it
            bar_arrive(&b.qd_empty[s]);
        }
        __syncwarp();
    }
    if (lane == 0) tma_store_wait_all();  // every reduction has landed before the CTA exits
    __syncwarp();
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTAs are dispatched in linear block order.  Non-causal: the key blocks
    // of one head are adjacent, so concurrent CTAs share that head's Q and dO
    // in L2.  Causal: heaviest first (key block j sees the query blocks from
    // first_qblock(j) on, fewer as j grows), so the short CTAs fill the tail.
    int j = blockIdx.x, bh = blockIdx.y;
    if (p.causal) {
        const long long lin = (long long)blockIdx.y * gridDim.x + blockIdx.x;
        j = (int)(lin / p.BH);
        bh = (int)(lin % p.BH);
    }
    const int i0 = first_qblock(p, j);
    const int nqb = p.n_qblocks - i0 > 0 ? p.n_qblocks - i0 : 0;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    BBars b;
    b.kv_full = bars;
    b.qd_full = bars + 1;
    b.qd_empty = bars + 3;
    b.s_full = bars + 5;
    b.ds_ready = bars + 6;
    b.dq_full = bars + 7;
    b.dq_empty = bars + 8;
    b.done = bars + 9;
    b.ld_full = bars + 10;
    b.ld_free = bars + 11;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

    if (threadIdx.x == 0) *skip = timeout_recorded(p.status) ? 1 : 0;
    __syncthreads();
    if (*skip) return;  // an earlier launch gave up: leave the device quiet

    if (threadIdx.x == 0) {
        bar_init(b.kv_full, 1);
        for (int s = 0; s < 2; ++s) {
            bar_init(&b.qd_full[s], 1);
            bar_init(&b.qd_empty[s], 5);
        }
        bar_init(b.s_full, 1);
        bar_init(b.ds_ready, 128);
        bar_init(b.dq_full, 1);
        bar_init(b.dq_empty, 128);
        bar_init(b.done, 1);
        bar_init(b.ld_full, 128);
        bar_init(b.ld_free, 128);
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

    if (warp >= 2 && warp < 6) {
        bwd_ds_role<D>(p, smem, b, abort_flag, tmem, bh, j, i0, nqb, warp & 3, lane);
    } else if (warp >= 6) {
        bwd_dq_role<D>(p, smem, b, abort_flag, tmem, bh, i0, nqb, warp & 3, lane);
    } else if (warp == 1) {
        if (lane == 0 && nqb > 0) {
            bwd_mma<D>(p, smem, b, abort_flag, tmem, nqb);
            tc_commit(b.done);  // every issued MMA finishes before tensor memory is released
            drain_wait(b.done, 0, p.status);
        }
        __syncwarp();
    } else {
        if (lane == 0 && nqb > 0) bwd_producer<D>(p, smem, b, abort_flag, bh, j, i0, nqb);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

// ---------------------------------------------------------------- d = 128: the pipelined main kernel
//
// The same five products with query blocks of 64 rows.  Two blocks' score
// tiles then fit in tensor memory beside dV and dK, so while the dS warpgroup
// works on block i the tensor core computes S^T and dP^T of block i + 1 and
// the dV, dK and dQ products of block i - 1.  dQ is computed transposed,
// dQ_i^T = K_j^T dS_i^T, with the head dims on the 128 TMEM lanes and the
// block's 64 queries in 64 columns; the dQ warpgroup has one thread per head
// dim.  K_j read MN-major (head dims along M) is the same shared-memory tile
// as for S^T, and dS_i (keys x queries, queries contiguous) serves as the
// MN-major B operand.  The dQ warpgroup stages its fp32 rows for the bulk
// reductions in a buffer of its own, so a Q / dO slot is free once the dV and
// dK products have read it: staged in the slot, as bwd_main does, the next
// loads would wait for the reductions to read the staging out.
//
// The CTAs are persistent, one per SM, each taking (batch*head, key block)
// units in turn; K_j and V_j are reloaded per unit (the next unit's pair is
// prefetched into L2 a few blocks before the switch), and the dQ warpgroup
// writes a unit's dV and dK while the next unit's first blocks run.
//
// Tensor memory, buffer b (the blocks i with i % 2 == b) at column 128 b:
//   +0..63 S^T, then P^T (bf16 pairs) in +0..31, then dQ_i^T in +0..63;
//   +64..127 dP^T, then dS^T in +64..95.   dV at 256, dK at 384.
// The products of one thread execute in issue order, so dQ_i^T may overwrite
// P^T right after the dV product that reads it.
struct PCfg {
    static constexpr int D = 128;
    static constexpr int QB = 64;                 // queries per block
    static constexpr int NQS = 3;                 // Q / dO slots
    static constexpr int KV_PANEL = 128 * 128;    // 128 key rows x 128 B
    static constexpr int KV_TILE = 2 * KV_PANEL;  // 128 keys x 128 dims bf16
    static constexpr int Q_PANEL = QB * 128;      // 64 rows x 128 B
    static constexpr int Q_TILE = 2 * Q_PANEL;    // 64 queries x 128 dims bf16
    static constexpr int SLOT = 2 * Q_TILE;       // Q_i then dO_i
    static constexpr int DS_TILE = 128 * 128;     // 128 keys x 64 queries bf16
    static constexpr int STG = 4 * 2 * 4096;      // dQ staging: 4 warps x 2 boxes of 32 rows x 32 fp32
    static constexpr uint32_t TM_DV = 256, TM_DK = 384, TM_COLS = 512;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KV_TILE;
    static constexpr int OFF_QD = OFF_V + KV_TILE;       // [NQS] slots
    static constexpr int OFF_DS = OFF_QD + NQS * SLOT;   // [2]
    static constexpr int OFF_STG = OFF_DS + 2 * DS_TILE;  // dQ staging, 8 KB per warp of the dQ warpgroup
    static constexpr int OFF_LD = OFF_STG + STG;          // [2] x (-lse2[64], -D[64])
    static constexpr int OFF_BAR = OFF_LD + 2 * 128 * 4;
    static constexpr int N_BARS = 2 + 2 * NQS + 4 * 2 + 4;
    static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t ID_S = idesc_make(128, QB, 1u, false, false);  // S^T, dP^T: 128 keys x 64 queries
    static constexpr uint32_t ID_G = idesc_make(128, D, 1u, false, true);   // dV, dK: B = dO_i / Q_i MN-major
    static constexpr uint32_t ID_DQT = idesc_make(128, QB, 1u, true, true);  // dQ^T: both operands MN-major
};

struct PBars {
    uint64_t* kv_full;    // K_j, V_j of the unit landed
    uint64_t* kv_empty;   // every product of the unit done: K_j, V_j may be replaced
    uint64_t* qd_full;    // [NQS]
    uint64_t* qd_empty;   // [NQS], the dV / dK products read the slot
    uint64_t* s_full;     // [2], S^T and dP^T of the buffer's block computed
    uint64_t* ds_ready;   // [2], 128 arrivals: P^T, dS^T in TMEM and dS in shared memory
    uint64_t* dq_full;    // [2], dQ_i^T computed (and everything issued before it)
    uint64_t* dq_empty;   // [2], 128 arrivals: dQ_i^T read out of TMEM
    uint64_t* acc_full;   // dV, dK of the unit final
    uint64_t* acc_empty;  // 128 arrivals: dV, dK read out of TMEM
    uint64_t* done;       // every product finished (before tensor memory is released)
    uint64_t* ld_full;    // 128 arrivals per block: its lse2 / D staged
};

// First 64-query block that sees key block j (see first_qblock).
__device__ __forceinline__ int first_qblock64(const BwdParams& p, int j) {
    if (!p.causal) return 0;
    const long long need = (long long)j * 128 - (p.Nk - p.Nq) - (PCfg::QB - 1);
    if (need <= 0) return 0;
    return (int)((need + PCfg::QB - 1) / PCfg::QB);
}

// A unit is one 128-key block j of one (batch, head).  Non-causal: the key
// blocks of a head adjacent, so CTAs running at the same time share its Q and
// dO in L2; causal: heaviest first (key block j sees the 64-query blocks from
// first_qblock64(j) on), so the short units fill the tail.
struct BUnit {
    int bh, j, i0, nqb;
};

__device__ __forceinline__ BUnit bwd_unit(const BwdParams& p, int u) {
    BUnit g;
    if (p.causal) {
        g.j = u / p.BH;
        g.bh = u - g.j * p.BH;
    } else {
        g.bh = u / p.n_kblocks;
        g.j = u - g.bh * p.n_kblocks;
    }
    g.i0 = first_qblock64(p, g.j);
    const int n_all = (p.Nq + PCfg::QB - 1) / PCfg::QB;
    g.nqb = n_all - g.i0 > 0 ? n_all - g.i0 : 0;
    return g;
}

// This CTA's next unit: rounds of gridDim.x units, every other round in
// reverse CTA order, or -1 when none is left.
__device__ __forceinline__ int bwd_next_unit(int n_units, int& round_) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    for (;;) {
        const long long base = (long long)round_ * G;
        if (base >= n_units) return -1;
        const int u = (int)base + ((round_ & 1) ? (G - 1 - c) : c);
        ++round_;
        if (u < n_units) return u;
    }
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Start pulling a box into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

constexpr int kPrefetchAhead = 3;  // 64-query blocks before a unit's end: the next unit's K/V to L2

__device__ void pipe_producer(const BwdParams& p, uint8_t* smem, const PBars& b, volatile int* abort_flag) {
    using C = PCfg;
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    tma_prefetch_map(&p.tm_do);
    const int n_units = p.BH * p.n_kblocks;
    int gq = 0, nu = 0, round_ = 0, peek_round = 0;
    bool ok = true;
    for (int u = bwd_next_unit(n_units, round_); ok && u >= 0; u = bwd_next_unit(n_units, round_)) {
        const BUnit g = bwd_unit(p, u);
        if (g.nqb == 0) continue;
        // K_j and V_j replace the previous unit's once all its products are done
        if (nu > 0 && !wait_bar(b.kv_empty, (uint32_t)((nu - 1) & 1), abort_flag, p.status)) break;
        bar_arrive_expect_tx(b.kv_full, 2 * C::KV_TILE);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn) {
            tma_load_3d(smem + C::OFF_K + pn * C::KV_PANEL, &p.tm_k, b.kv_full, pn * 64, g.j * 128, g.bh);
            tma_load_3d(smem + C::OFF_V + pn * C::KV_PANEL, &p.tm_v, b.kv_full, pn * 64, g.j * 128, g.bh);
        }
        peek_round = round_;
        const int un = bwd_next_unit(n_units, peek_round);
        ++nu;
        for (int it = 0; it < g.nqb; ++it, ++gq) {
            // A few blocks before the unit ends the next unit's K and V start
            // towards L2, so that their load at the unit boundary hits there
            // (issued earlier, the streams of Q, dO and the dQ reductions
            // evict them again).
            if (un >= 0 && it == (g.nqb > kPrefetchAhead ? g.nqb - kPrefetchAhead : 0)) {
                const BUnit gn = bwd_unit(p, un);
#pragma unroll
                for (int pn = 0; pn < 2; ++pn) {
                    tma_prefetch_l2_3d(&p.tm_k, pn * 64, gn.j * 128, gn.bh);
                    tma_prefetch_l2_3d(&p.tm_v, pn * 64, gn.j * 128, gn.bh);
                }
            }
            const int s = gq % C::NQS;
            if (gq >= C::NQS && !wait_bar(&b.qd_empty[s], (uint32_t)((gq / C::NQS - 1) & 1), abort_flag, p.status)) {
                ok = false;
                break;
            }
            const int i = g.i0 + it;
            uint8_t* slot = smem + C::OFF_QD + s * C::SLOT;
            bar_arrive_expect_tx(&b.qd_full[s], C::SLOT);
#pragma unroll
            for (int pn = 0; pn < 2; ++pn) {
                tma_load_3d(slot + pn * C::Q_PANEL, &p.tm_q, &b.qd_full[s], pn * 64, i * C::QB, g.bh);
                tma_load_3d(slot + C::Q_TILE + pn * C::Q_PANEL, &p.tm_do, &b.qd_full[s], pn * 64, i * C::QB, g.bh);
            }
        }
    }
    // every copy started here lands before the CTA exits
    if (nu > 0) drain_wait(b.kv_full, (uint32_t)((nu - 1) & 1), p.status);
    for (int q = gq - C::NQS > 0 ? gq - C::NQS : 0; q < gq; ++q)
        drain_wait(&b.qd_full[q % C::NQS], (uint32_t)((q / C::NQS) & 1), p.status);
}

// One thread.  Per unit, step it issues S^T, dP^T of block it into buffer
// (global block) % 2 once dQ^T of the block two before has left it, then the
// dV, dK and dQ^T products of block it - 1 once its dS is ready; a last step
// issues those of the unit's final block.  Block counters run on across units.
__device__ void pipe_mma(const BwdParams& p, uint8_t* smem, const PBars& b, volatile int* abort_flag,
                         uint32_t tmem) {
    using C = PCfg;
    const uint32_t sb = smem_u32(smem);
    const uint64_t k_kmaj = sdesc_sw128(sb + C::OFF_K, 16, 1024);
    const uint64_t v_kmaj = sdesc_sw128(sb + C::OFF_V, 16, 1024);
    const uint64_t k_mn = sdesc_sw128(sb + C::OFF_K, C::KV_PANEL, 1024);  // K_j^T: head dims along M
    constexpr int KVP = C::KV_PANEL >> 4, QP = C::Q_PANEL >> 4;           // panel strides, descriptor units
    const int n_units = p.BH * p.n_kblocks;
    int gb = 0, nu = 0, round_ = 0;
    for (int u = bwd_next_unit(n_units, round_); u >= 0; u = bwd_next_unit(n_units, round_)) {
        const BUnit g = bwd_unit(p, u);
        if (g.nqb == 0) continue;
        if (!wait_bar(b.kv_full, (uint32_t)(nu & 1), abort_flag, p.status)) return;
        for (int it = 0; it <= g.nqb; ++it) {
            if (it < g.nqb) {
                const int q = gb + it, s = q % C::NQS, bf = q & 1;
                const uint32_t q_addr = sb + C::OFF_QD + s * C::SLOT, do_addr = q_addr + C::Q_TILE;
                if (!wait_bar(&b.qd_full[s], (uint32_t)((q / C::NQS) & 1), abort_flag, p.status)) return;
                if (q >= 2 && !wait_bar(&b.dq_empty[bf], (uint32_t)(((q - 2) >> 1) & 1), abort_flag, p.status))
                    return;
                tc_fence_after();
                const uint32_t t_s = tmem + 128u * (uint32_t)bf;
                // S^T = K_j Q_i^T, dP^T = V_j dO_i^T: 8 steps of 16 head dims (32 bytes);
                // K and V advance a 16 KB panel every 4 steps, Q and dO an 8 KB one
                const uint64_t qd = sdesc_sw128(q_addr, 16, 1024), dd = sdesc_sw128(do_addr, 16, 1024);
                mma4_ss<2, 4, 6, 2, 4, 6, false>(t_s, k_kmaj, qd, C::ID_S, 0u);
                mma4_ss<2, 4, 6, 2, 4, 6, false>(t_s, k_kmaj + KVP, qd + QP, C::ID_S, 1u);
                mma4_ss<2, 4, 6, 2, 4, 6, false>(t_s + 64, v_kmaj, dd, C::ID_S, 0u);
                mma4_ss<2, 4, 6, 2, 4, 6, false>(t_s + 64, v_kmaj + KVP, dd + QP, C::ID_S, 1u);
                tc_commit(&b.s_full[bf]);
            }
            if (it >= 1) {
                const int q = gb + it - 1, s = q % C::NQS, bf = q & 1;
                const uint32_t q_addr = sb + C::OFF_QD + s * C::SLOT, do_addr = q_addr + C::Q_TILE;
                if (!wait_bar(&b.ds_ready[bf], (uint32_t)((q >> 1) & 1), abort_flag, p.status)) return;
                // the unit's first dV / dK product overwrites the accumulators:
                // the previous unit's must have been read out
                if (it == 1 && nu > 0 &&
                    !wait_bar(b.acc_empty, (uint32_t)((nu - 1) & 1), abort_flag, p.status))
                    return;
                tc_fence_after();
                const uint32_t t_s = tmem + 128u * (uint32_t)bf;
                // dV += P^T dO_i, dK += dS^T Q_i: 4 steps of 16 queries (8 TMEM columns of bf16
                // pairs; the MN-major B advances 16 rows, 2 KB)
                mma4_ts<8, 16, 24, 128, 256, 384, false>(tmem + C::TM_DV, t_s, sdesc_sw128(do_addr, C::Q_PANEL, 1024),
                                                         C::ID_G, it > 1 ? 1u : 0u);
                mma4_ts<8, 16, 24, 128, 256, 384, false>(tmem + C::TM_DK, t_s + 64,
                                                         sdesc_sw128(q_addr, C::Q_PANEL, 1024), C::ID_G,
                                                         it > 1 ? 1u : 0u);
                tc_commit(&b.qd_empty[s]);
                if (it == g.nqb) tc_commit(b.acc_full);
                // dQ_i^T = K_j^T dS_i^T: 8 steps of 16 keys, both operands advance 16 rows (2 KB)
                const uint64_t dsd = sdesc_sw128(sb + C::OFF_DS + bf * C::DS_TILE, C::DS_TILE, 1024);
                mma4_ss<128, 256, 384, 128, 256, 384, false>(t_s, k_mn, dsd, C::ID_DQT, 0u);
                mma4_ss<128, 256, 384, 128, 256, 384, false>(t_s, k_mn + 512, dsd + 512, C::ID_DQT, 1u);
                tc_commit(&b.dq_full[bf]);
            }
        }
        tc_commit(b.kv_empty);  // K_j, V_j read by every product of the unit
        gb += g.nqb;
        ++nu;
    }
}

// One thread per key row (TMEM lane): P^T and dS^T of each 64-query block of
// every unit.
__device__ void pipe_ds_role(const BwdParams& p, uint8_t* smem, const PBars& b, volatile int* abort_flag,
                             uint32_t tmem, int wq, int lane) {
    using C = PCfg;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int off = p.Nk - p.Nq;
    const float cs = p.c_scale;
    float* lds = reinterpret_cast<float*>(smem + C::OFF_LD);  // [2][128]: -lse2 of the block's queries, then -D
    const int n_units = p.BH * p.n_kblocks;
    int gb = 0, round_ = 0;
    bool ok = true;
    for (int u = bwd_next_unit(n_units, round_); ok && u >= 0; u = bwd_next_unit(n_units, round_)) {
        const BUnit g = bwd_unit(p, u);
        const int key = g.j * 128 + row;
        const bool key_ok = key < p.Nk;
        // this thread's entry of each block -- lse2 (rows 0-63) or D (64-127) -- loaded a block ahead
        const float* src = (row < C::QB ? p.lse2 + row : p.dvec + (row - C::QB)) + (size_t)g.bh * p.nq_pad +
                           (size_t)g.i0 * C::QB;
        float nx = g.nqb > 0 ? src[0] : 0.f;
        for (int it = 0; it < g.nqb; ++it) {
            const int q = gb + it, i = g.i0 + it, bf = q & 1;
            const float mine = nx;
            if (it + 1 < g.nqb) nx = src[(size_t)(it + 1) * C::QB];
            // Buffer bf held the entries of the block two before: every thread
            // finished that block before it arrived for the previous one, which
            // this thread has seen.
            lds[bf * 128 + row] = -mine;  // negated: the score step is one fma, the dS step one add
            bar_arrive(b.ld_full);
            ok = __all_sync(0xffffffffu, wait_bar(b.ld_full, (uint32_t)(q & 1), abort_flag, p.status));
            if (!ok) break;
            // S^T, dP^T ready; their commit also covers dQ^T of the block two
            // before, the last reader of dS buffer bf
            ok = __all_sync(0xffffffffu, wait_bar(&b.s_full[bf], (uint32_t)((q >> 1) & 1), abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = tmem + lane_off + 128u * (uint32_t)bf, tP = tS + 64;
            const uint32_t ds_row = smem_u32(smem + C::OFF_DS + bf * C::DS_TILE) + (uint32_t)(row * 128);
            // Queries of this block before `vis_from` do not see this key (causal
            // mask); the whole warp takes the mask-free path when none of its keys
            // needs it.  Scores, shifts and products run as packed pairs.
            const int vis_from = key_ok ? (p.causal ? key - off - i * C::QB : 0) : C::QB;
            const bool all_visible = __all_sync(0xffffffffu, vis_from <= 0);
            const float* nl = lds + bf * 128;  // -lse2 of the block's queries
            const float* nd = nl + C::QB;      // -D
            const uint64_t cs2 = f2_pack(cs, cs);
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {  // 32 queries per chunk
                uint32_t sv[32], dp[32];
                tmem_ld32(tS + 32 * c, sv);
                tmem_ld32(tP + 32 * c, dp);
                tmem_ld_wait();
                reg_after_wait<32>(sv);
                reg_after_wait<32>(dp);
                uint32_t pw[16], dw[16];
#pragma unroll
                for (int t4 = 0; t4 < 8; ++t4) {
                    const float4 L = *reinterpret_cast<const float4*>(nl + 32 * c + 4 * t4);
                    const float4 Dn = *reinterpret_cast<const float4*>(nd + 32 * c + 4 * t4);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int t = 4 * t4 + 2 * h;
                        const uint64_t x = f2_fma(f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1])), cs2,
                                                  h ? f2_pack(L.z, L.w) : f2_pack(L.x, L.y));
                        float p0, p1;
                        f2_unpack(x, p0, p1);
                        p0 = ex2(p0);
                        p1 = ex2(p1);
                        if (!all_visible) {
                            const int tq = 32 * c + t;  // query index within the block
                            p0 = tq >= vis_from ? p0 : 0.f;
                            p1 = tq + 1 >= vis_from ? p1 : 0.f;
                        }
                        const uint64_t pp = f2_pack(p0, p1);
                        const uint64_t diff = f2_add(f2_pack(__uint_as_float(dp[t]), __uint_as_float(dp[t + 1])),
                                                     h ? f2_pack(Dn.z, Dn.w) : f2_pack(Dn.x, Dn.y));
                        float d0, d1;
                        f2_unpack(f2_mul(pp, diff), d0, d1);
                        pw[2 * t4 + h] = pack_bf16(p0, p1);
                        dw[2 * t4 + h] = pack_bf16(d0, d1);
                    }
                }
                tmem_st16(tS + 16 * c, pw);
                tmem_st16(tP + 16 * c, dw);
                // dS row `row`, queries 32c..32c+31: 16-byte chunks 4c..4c+3 of the
                // 128-byte row, 128-byte swizzle (chunk ^ row % 8)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t chunk = (uint32_t)(4 * c + k) ^ (uint32_t)(row & 7);
                    st_shared_v4(ds_row + chunk * 16u, dw[4 * k], dw[4 * k + 1], dw[4 * k + 2], dw[4 * k + 3]);
                }
            }
            tmem_st_wait();
            fence_async_smem();
            tc_fence_before();
            bar_arrive(&b.ds_ready[bf]);
        }
        gb += g.nqb;
    }
}

// dV and scale * dK rows of one unit's key block -> bf16 (one thread per key
// row, i.e. TMEM lane); zeros when no query sees the block.
__device__ __forceinline__ bool pipe_epilogue(const BwdParams& p, const PBars& b, volatile int* abort_flag,
                                              uint32_t tmem, const BUnit& g, int nu, int row, uint32_t lane_off) {
    using C = PCfg;
    constexpr int D = C::D;
    const int key = g.j * 128 + row;
    if (g.nqb > 0) {
        if (!__all_sync(0xffffffffu, wait_bar(b.acc_full, (uint32_t)(nu & 1), abort_flag, p.status))) return false;
        tc_fence_after();
    }
    uint16_t* dvr = p.dv + ((size_t)g.bh * p.Nk + key) * D;
    uint16_t* dkr = p.dk + ((size_t)g.bh * p.Nk + key) * D;
    const float sc = p.scale;
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t a[32], gk[32];
        if (g.nqb > 0) {
            tmem_ld32(tmem + lane_off + C::TM_DV + 32 * ch, a);
            tmem_ld32(tmem + lane_off + C::TM_DK + 32 * ch, gk);
            tmem_ld_wait();
            reg_after_wait<32>(a);
            reg_after_wait<32>(gk);
            if (ch == D / 32 - 1) {  // the accumulators are free for the next unit
                tc_fence_before();
                bar_arrive(b.acc_empty);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = gk[e] = 0u;
        }
        if (key < p.Nk) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
                st_global_v4(dvr + 32 * ch + e, pack_bf16(__uint_as_float(a[e]), __uint_as_float(a[e + 1])),
                             pack_bf16(__uint_as_float(a[e + 2]), __uint_as_float(a[e + 3])),
                             pack_bf16(__uint_as_float(a[e + 4]), __uint_as_float(a[e + 5])),
                             pack_bf16(__uint_as_float(a[e + 6]), __uint_as_float(a[e + 7])));
                st_global_v4(dkr + 32 * ch + e,
                             pack_bf16(__uint_as_float(gk[e]) * sc, __uint_as_float(gk[e + 1]) * sc),
                             pack_bf16(__uint_as_float(gk[e + 2]) * sc, __uint_as_float(gk[e + 3]) * sc),
                             pack_bf16(__uint_as_float(gk[e + 4]) * sc, __uint_as_float(gk[e + 5]) * sc),
                             pack_bf16(__uint_as_float(gk[e + 6]) * sc, __uint_as_float(gk[e + 7]) * sc));
            }
        }
    }
    return true;
}

// dQ warpgroup: per block one thread per head dim (TMEM lane of dQ_i^T), the
// block's 64 dQ values added into the accumulator; after a unit's last block,
// one thread per key row for its dV, dK epilogue.
__device__ void pipe_dq_role(const BwdParams& p, uint8_t* smem, const PBars& b, volatile int* abort_flag,
                             uint32_t tmem, int wq, int lane) {
    using C = PCfg;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;  // head dims (dQ^T) or key rows (dV, dK) 32 wq ..
    if (lane == 0) tma_prefetch_map(&p.tm_dq);
    uint8_t* stage_p = smem + C::OFF_STG + wq * 8192;
    const uint32_t stage = smem_u32(stage_p) + (uint32_t)((lane & 3) * 4);
    const int n_units = p.BH * p.n_kblocks;
    int gb = 0, nu = 0, round_ = 0;
    bool ok = true;
    for (int u = bwd_next_unit(n_units, round_); ok && u >= 0; u = bwd_next_unit(n_units, round_)) {
        const BUnit g = bwd_unit(p, u);
        for (int it = 0; it < g.nqb; ++it) {
            const int q = gb + it, bf = q & 1;
            ok = __all_sync(0xffffffffu, wait_bar(&b.dq_full[bf], (uint32_t)((q >> 1) & 1), abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[C::QB];  // this head dim of the block's 64 queries
            tmem_ld32(tmem + lane_off + 128u * (uint32_t)bf, v);
            tmem_ld32(tmem + lane_off + 128u * (uint32_t)bf + 32, v + 32);
            tmem_ld_wait();
            reg_after_wait<C::QB>(v);
            tc_fence_before();
            bar_arrive(&b.dq_empty[bf]);
            // Stage the warp's 32 head dims x 64 queries as two boxes of 32 query
            // rows x 32 fp32 (128-byte rows, 128-byte swizzle: 16-byte chunk k of
            // row r at k ^ (r % 8)) once the engine has read the previous block's,
            // then let the bulk-copy engine add them into the accumulator.
            if (lane == 0) tma_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int qq = 0; qq < C::QB; ++qq)
                st_shared_b32(stage + (uint32_t)((qq >> 5) * 4096 + (qq & 31) * 128) +
                                  ((((uint32_t)lane >> 2) ^ (uint32_t)(qq & 7)) << 4),
                              v[qq]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int row0 = (g.i0 + it) * C::QB;
                tma_reduce_add_3d(&p.tm_dq, stage_p, wq * 32, row0, g.bh);
                tma_reduce_add_3d(&p.tm_dq, stage_p + 4096, wq * 32, row0 + 32, g.bh);
                tma_store_commit();
            }
            __syncwarp();
        }
        if (!ok) break;
        ok = pipe_epilogue(p, b, abort_flag, tmem, g, nu, wq * 32 + lane, lane_off);
        gb += g.nqb;
        nu += g.nqb > 0;
    }
    if (lane == 0) tma_store_wait_all();  // every reduction has landed before the CTA exits
    __syncwarp();
}

// Persistent: one CTA per SM takes (batch*head, key block) units in snake
// order; K_j and V_j are reloaded per unit, the dV / dK epilogue of a unit
// runs while the next unit's first blocks are computed.
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_pipe_kernel(const __grid_constant__ BwdParams p) {
    using C = PCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    PBars b;
    b.kv_full = bars;
    b.kv_empty = bars + 1;
    b.qd_full = bars + 2;
    b.qd_empty = b.qd_full + C::NQS;
    b.s_full = b.qd_empty + C::NQS;
    b.ds_ready = b.s_full + 2;
    b.dq_full = b.ds_ready + 2;
    b.dq_empty = b.dq_full + 2;
    b.acc_full = b.dq_empty + 2;
    b.acc_empty = b.acc_full + 1;
    b.done = b.acc_empty + 1;
    b.ld_full = b.done + 1;
    static_assert(2 + 2 * PCfg::NQS + 8 + 4 == PCfg::N_BARS, "barrier count");
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

    if (threadIdx.x == 0) *skip = timeout_recorded(p.status) ? 1 : 0;
    __syncthreads();
    if (*skip) return;  // an earlier launch gave up: leave the device quiet

    if (threadIdx.x == 0) {
        bar_init(b.kv_full, 1);
        bar_init(b.kv_empty, 1);
        for (int s = 0; s < C::NQS; ++s) {
            bar_init(&b.qd_full[s], 1);
            bar_init(&b.qd_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            bar_init(&b.s_full[t], 1);
            bar_init(&b.ds_ready[t], 128);
            bar_init(&b.dq_full[t], 1);
            bar_init(&b.dq_empty[t], 128);
        }
        bar_init(b.acc_full, 1);
        bar_init(b.acc_empty, 128);
        bar_init(b.done, 1);
        bar_init(b.ld_full, 128);
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

    if (warp >= 2 && warp < 6) {
        pipe_ds_role(p, smem, b, abort_flag, tmem, warp & 3, lane);
    } else if (warp >= 6) {
        pipe_dq_role(p, smem, b, abort_flag, tmem, warp & 3, lane);
    } else if (warp == 1) {
        if (lane == 0) {
            pipe_mma(p, smem, b, abort_flag, tmem);
            tc_commit(b.done);  // every issued MMA finishes before tensor memory is released
            drain_wait(b.done, 0, p.status);
        }
        __syncwarp();
    } else {
        if (lane == 0) pipe_producer(p, smem, b, abort_flag);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

cudaError_t launch_bwd_pipe(const BwdParams& p, int sm_count, cudaStream_t stream) {
    using C = PCfg;
    const long long prep_warps = (long long)p.BH * p.nq_pad;
    bwd_prep_kernel<128><<<(unsigned)((prep_warps + 7) / 8), 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long n_units = (long long)p.BH * p.n_kblocks;
    const int grid = (int)(n_units < sm_count ? n_units : sm_count);
    bwd_pipe_kernel<<<grid, kBwdThreads, C::SMEM_BYTES, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long dq_warps = (long long)p.BH * p.Nq;
    bwd_dq_kernel<128><<<(unsigned)((dq_warps + 7) / 8), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, cudaStream_t stream) {
    using C = BCfg<D>;
    const long long prep_warps = (long long)p.BH * p.nq_pad;
    bwd_prep_kernel<D><<<(unsigned)((prep_warps + 7) / 8), 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    bwd_main_kernel<D><<<dim3((unsigned)p.n_kblocks, (unsigned)p.BH), kBwdThreads, C::SMEM_BYTES, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long dq_warps = (long long)p.BH * p.Nq;
    bwd_dq_kernel<D><<<(unsigned)((dq_warps + 7) / 8), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(int BH, int Nq, int d) {
    const size_t nq_pad = ((size_t)Nq + 127) / 128 * 128;
    return (size_t)BH * nq_pad * ((size_t)d + 2) * sizeof(float);
}

cudaError_t launch_bwd(int d, const BwdParams& p, int sm_count, cudaStream_t stream) {
    if (d == 128) return launch_bwd_pipe(p, sm_count, stream);
    if (d == 64) return launch_bwd_d<64>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
