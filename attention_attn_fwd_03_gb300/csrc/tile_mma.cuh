// tile_mma.cuh -- the two GEMMs of one attention block on tcgen05, shared by
// the dense prefill kernel and the paged kernel.
//
// Operand layout (both kernels stage tiles the same way):
//   Q and K tiles: 128 rows, K-major, 128-byte swizzle, split into panels of
//   128 bytes of the head dim (64 bf16 or 128 e4m3 elements); a panel is
//   128 rows x 128 B = 16 KB and panel p of a tile starts p * 16 KB in.
//   V tiles: the same bytes read MN-major (the head dim is the N axis).
//   S: tensor memory, 128 lanes x 128 columns.  P, in the paged kernel and
//   the turn-based prefill kernel, overwrites S in tensor memory (bf16 pairs
//   or e4m3 quadruples per 32-bit column); in the decoupled prefill kernel P
//   is a shared-memory tile laid out like Q (128 rows, K-major, 128-byte
//   swizzle, panels of 128 bytes of keys).
#pragma once

#include "ptx.cuh"

namespace attn {

template <int D, bool FP8>
struct TileMma {
    static constexpr int EB = FP8 ? 1 : 2;         // bytes per input element
    static constexpr int PANEL = 128 / EB;         // elements in one 128-byte row panel
    static constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B
    static constexpr int MMA_K = FP8 ? 32 : 16;    // K per tcgen05.mma (32 bytes)
    static constexpr int S_STEPS = D / MMA_K;
    static constexpr int PV_STEPS = 128 / MMA_K;
    static constexpr uint32_t P_STEP_COLS = MMA_K * EB / 4;  // TMEM columns per PV step
    static constexpr uint32_t FMT = FP8 ? 0u : 1u;           // e4m3 / bf16
    static constexpr uint32_t ID_S = idesc_make(128, 128, FMT, false, false);
    static constexpr uint32_t ID_PV = idesc_make(128, D, FMT, false, true);
};

// S = Q K^T: S_STEPS MMAs along d.  a0 / b0 are the descriptors of the Q and K
// tiles; the k-th step starts (k / 4) panels and (k % 4) * 32 bytes further
// (the descriptor's start-address field holds byte address >> 4).
template <int D, bool FP8>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t a0, uint64_t b0) {
    using C = TileMma<D, FP8>;
    // four 32-byte K steps per 128-byte panel; next panel PANEL_BYTES further
#pragma unroll
    for (int g = 0; g < C::S_STEPS / 4; ++g) {
        const uint64_t po = (uint64_t)((g * C::PANEL_BYTES) >> 4);
        mma4_ss<2, 4, 6, 2, 4, 6, FP8>(d_tmem, a0 + po, b0 + po, C::ID_S, g > 0 ? 1u : 0u);
    }
}

// O += P V: PV_STEPS MMAs along the keys; P from tensor memory (P_STEP_COLS
// columns per step), b0 the descriptor of the MN-major V tile (step s starts
// s * MMA_K rows, i.e. s * MMA_K * 128 bytes, further).
template <int D, bool FP8>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t b0, bool accumulate) {
    using C = TileMma<D, FP8>;
    constexpr int PC = (int)C::P_STEP_COLS;
    constexpr int VB = (C::MMA_K * 128) >> 4;
#pragma unroll
    for (int g = 0; g < C::PV_STEPS / 4; ++g)
        mma4_ts<PC, 2 * PC, 3 * PC, VB, 2 * VB, 3 * VB, FP8>(o_tmem, p_tmem + (uint32_t)(4 * g * PC),
                                                           b0 + (uint64_t)(4 * g * VB), C::ID_PV,
                                                           (accumulate || g > 0) ? 1u : 0u);
}

// O += P V with P in shared memory (the decoupled prefill kernel): A = P, K-major like
// a Q tile (panels of 128 bytes of keys, PANEL_BYTES apart), B = V MN-major.
// Step s covers keys s * MMA_K ..: A advances (s % 4) * 32 bytes within a
// panel and a panel every 4 steps; B advances s * MMA_K rows.
template <int D, bool FP8>
__device__ __forceinline__ void issue_pv_ss(uint32_t o_tmem, uint64_t a0, uint64_t b0, bool accumulate) {
    using C = TileMma<D, FP8>;
    constexpr int VB = (C::MMA_K * 128) >> 4;
#pragma unroll
    for (int g = 0; g < C::PV_STEPS / 4; ++g) {
        const uint64_t po = (uint64_t)((g * C::PANEL_BYTES) >> 4);
        mma4_ss<2, 4, 6, VB, 2 * VB, 3 * VB, FP8>(o_tmem, a0 + po, b0 + (uint64_t)(4 * g * VB), C::ID_PV,
                                                 (accumulate || g > 0) ? 1u : 0u);
    }
}

}  // namespace attn
