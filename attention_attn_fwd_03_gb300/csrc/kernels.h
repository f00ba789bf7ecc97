// kernels.h -- parameter blocks and launchers shared between the C-ABI layer
// (api.cu) and the kernel translation units (prefill.cu, decode.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn {

// Dense prefill.  Q/K/V are described by 3-D TMA maps over (d, rows, B*H)
// with a (128 bytes, 128 rows) box, 128-byte swizzle and zero fill; O by a
// map with a (32 elements, 32 rows) box and no swizzle (per-warp stores).
struct PrefillParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tm_o;
    float* lse;         // [B*H, Nq] or nullptr
    unsigned* status;   // device status word (bit mask of ATTN_ERR_* codes)
    int BH, Nq, Nk, causal;
    int n_pairs;        // ceil(Nq / 256): a work unit is two 128-row query tiles
    int n_units;        // n_pairs * B * H
    float c_scale;      // scale * log2(e) [* q_descale * k_descale]
    float o_scale;      // 1 [or v_descale]
};

constexpr int kPrefillThreads = 352;  // 2 MMA issuer warps + TMA warp + 2 softmax warpgroups

int prefill_smem_bytes(int d, bool fp8);
// grid = number of persistent CTAs (at most one per SM and at most n_units)
cudaError_t launch_prefill(int d, bool fp8, const PrefillParams& p, int grid, cudaStream_t stream);

// Paged decode: split kernel writes per-split partials, merge kernel combines.
struct DecodeParams {
    const uint16_t* q;        // bf16 [B, H, d]
    const uint16_t* k_cache;  // bf16 [num_pages, page_size, H, d]
    const uint16_t* v_cache;
    const int32_t* block_table;  // [B, max_pages]
    const int32_t* seq_lens;     // [B]
    float* part_o;            // [B, H, max_splits, d]  unnormalised partial O
    float* part_ml;           // [B, H, max_splits, 2]  (m in log2 units, l)
    uint16_t* o;              // bf16 [B, H, d]
    float* lse;               // [B, H] or nullptr
    unsigned* status;
    int B, H, page_size, max_pages, num_pages;
    int pages_per_split, max_splits;
    float c_scale;            // scale * log2(e)
};

// Split plan shared by the size query and the launcher.
struct DecodePlan {
    int pages_per_split;
    int max_splits;
    size_t part_o_bytes;
    size_t part_ml_bytes;
    size_t workspace_bytes;
};
DecodePlan decode_plan(int B, int H, int d, int page_size, int max_pages);

cudaError_t launch_paged_decode(int d, const DecodeParams& p, cudaStream_t stream);

}  // namespace attn

#include "attn.h"

namespace attn {

// Device address of the calling device's status word (api.cu).
attn_status_t status_word_address(unsigned** out);

}  // namespace attn
