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
// Ragged mode: the same boxes over token-major tensors, dims (d, rows, heads)
// with a row stride of heads * d * 2 bytes; K/V boxes are R rows high.
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
    // ---- ragged mode only (variable-length sequences, keys contiguous or paged)
    const int4* units;       // 2 int4 per listed unit: (s, pair, h, q_start), (q_len, kv_len, kv_start, 0)
    const int* n_listed;     // number of listed units (written by the schedule pass)
    const int32_t* block_table;  // [B, max_pages] page ids; nullptr: contiguous keys from row kv_start
    uint16_t* o;             // bf16 [total_q, H, d] (rows of a tile that straddles a sequence end)
    int H, G;                // query heads, query heads per KV head
    int page_size, max_pages, num_pages;
    int rows_per_box;        // key rows per TMA box: min(page_size, 128), or 128 for contiguous keys
    int kv_rows;             // rows of the key tensor: the first row past it reads as zeros
};

constexpr int kPrefillThreads = 352;  // 2 MMA issuer warps + TMA warp + 2 softmax warpgroups (both designs)

// Turn-based prefill kernel (prefill.cu): P overwrites S in tensor memory.
int prefill_smem_bytes(int d, bool fp8);
// grid = number of persistent CTAs (at most one per SM and at most n_units)
cudaError_t launch_prefill(int d, bool fp8, const PrefillParams& p, int grid, cudaStream_t stream);
// Decoupled prefill kernel (prefill_sp.cu): P in shared memory, S of the next
// block computed during the softmax; the faster one for long rows.  Dense
// (non-ragged) launches only; same parameters and grid rule.
int prefill_sp_smem_bytes(int d, bool fp8);
cudaError_t launch_prefill_sp(int d, bool fp8, const PrefillParams& p, int grid, cudaStream_t stream);

// Ragged prefill: the prefill kernel over variable-length sequences of
// token-major tensors (q, o [total_q, H, d]; keys [rows, H_kv, d], contiguous
// per sequence or gathered through a block table).  A one-CTA schedule pass
// lists the units (sequence, query-tile pair, head), longest first.
struct RaggedSched {
    const int32_t* cu_q;      // [B + 1] query offsets
    const int32_t* seq_lens;  // [B] key counts (paged keys), or nullptr
    const int32_t* cu_k;      // [B + 1] key offsets (contiguous keys), or nullptr
    int4* units;              // out: 2 int4 per unit
    int* n_listed;            // out
    unsigned* status;
    int B, H, total_q, max_q_len, kv_cap, causal;  // kv_cap: largest valid key count (paged) or key rows
    int kv_bytes_per_key;     // K and V bytes of one key position (H_kv * d * 2 * 2)
};
// bytes of workspace the ragged path needs for these sizes (unit list + count)
size_t ragged_workspace_bytes(int B, int max_q_len, int H);
cudaError_t launch_ragged_prefill(int d, const RaggedSched& sp, const PrefillParams& p, int grid,
                                  cudaStream_t stream);

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

// Paged attention on the tensor cores (grouped-query decode, prefill chunks
// over a paged cache).  A query tile packs T tokens x G query heads of one KV
// head into its 128 rows (row = t * G + g).
struct PagedParams {
    CUtensorMap tm_q;  // q [total_q, H, d]: dims (d, H, total_q), box (64, G, T), 128-B swizzle
    CUtensorMap tm_k;  // cache [num_pages * page_size, H_kv, d]: dims (d, H_kv, slots), box (64, 1, R)
    CUtensorMap tm_v;
    const int32_t* block_table;  // [B, max_pages]
    const int32_t* cu_q;         // [B + 1] token offsets, or nullptr: one token per request
    const int32_t* seq_lens;     // [B] keys per request (paged)
    const int32_t* cu_k;         // [B + 1] key offsets into contiguous K/V, or nullptr: paged
    uint16_t* o;                 // bf16 [total_q, H, d]
    float* lse;                  // [total_q, H] or nullptr
    float* part_o;               // [total_q * H, n_splits, d] unnormalised partial O (n_splits > 1)
    float* part_ml;              // [total_q * H, n_splits, 2] (m in log2 units, l)
    unsigned* status;
    int* sched;                  // [0] fetch counter, [1] list length (written by the schedule pass)
    int* whole;                  // [B] or nullptr: 1 where the request's units cover all its keys (no merge)
    int4* sched_list;            // [n_units] units with work: (unit, q_start, q_len, kv_len)
    int B, H, H_kv, G, T;        // T = tokens per query tile
    int total_q, max_q_len, n_qt;
    int page_size, max_pages, num_pages, rows_per_box;  // rows_per_box = min(page_size, 128)
    int kv_rows;                 // rows of the K/V tensor maps (slots, or total_k): past them reads zeros
    int causal;
    int n_splits, split_blocks;  // split s covers KV blocks [s, s + 1) * split_blocks
    int n_units;                 // B * H_kv * n_qt * n_splits
    uint32_t q_tile_bytes;       // bytes one Q tile load delivers
    float c_scale;               // scale * log2(e)
    int n_ctas;                  // CTAs of the paged kernel (its persistent grid)
};

constexpr int kPagedThreads = 192;  // TMA warp + MMA warp + one softmax warpgroup

// Split plan shared by the size query and the launcher.
struct PagedPlan {
    int G, T, n_qt, n_splits, split_blocks;
    long long n_units;
    size_t list_offset;                  // byte offset of the unit list (after the 256-byte header)
    size_t part_o_bytes, part_ml_bytes;  // 0 when every unit covers all of its keys
    size_t whole_offset;                 // byte offset of the per-request whole flags, 0: none
    size_t part_o_offset, part_ml_offset;
    size_t workspace_bytes;              // header + list + partials
};
PagedPlan paged_plan(int total_q, int max_q_len, int B, int H, int H_kv, int d, int page_size, int max_pages);

int paged_smem_bytes(int d);
cudaError_t launch_paged(int d, const PagedParams& p, int grid, cudaStream_t stream);

// Failure-handling test: a bounded wait that nothing completes (selftest.cu).
cudaError_t launch_selftest_timeout(unsigned* status, cudaStream_t stream);
// Tensor-core rate check: n_ctas CTAs (one per SM), each timing 4 * n_groups
// back-to-back 128x128x16 bf16 MMAs into cycles[cta] (selftest.cu).
cudaError_t launch_selftest_mma_rate(int n_ctas, int n_groups, unsigned long long* cycles, unsigned* status,
                                     cudaStream_t stream);

// Backward: gradients of dense attention by recomputation from the LSE.
struct BwdParams {
    CUtensorMap tm_q;   // bf16 [BH, Nq, d], operand boxes as for prefill
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tm_do;  // dO, like q
    CUtensorMap tm_dq;  // fp32 dQ accumulator [BH, nq_pad, d]: box (32, 32, 1), 128-byte swizzle
    const uint16_t* o;     // bf16 [BH, Nq, d] forward output
    const uint16_t* dout;  // bf16 [BH, Nq, d]
    const float* lse;      // [BH, Nq] natural-log LSE from the forward pass
    float* lse2;           // [BH, nq_pad] lse * log2(e), +inf where no key is visible / padding
    float* dvec;           // [BH, nq_pad] rowsum(dO * O)
    float* dq_acc;         // [BH, nq_pad, d] fp32 dQ accumulator (unscaled)
    uint16_t* dq;          // bf16 [BH, Nq, d]
    uint16_t* dk;          // bf16 [BH, Nk, d]
    uint16_t* dv;          // bf16 [BH, Nk, d]
    unsigned* status;
    int BH, Nq, Nk, causal;
    int n_qblocks, n_kblocks, nq_pad;
    float c_scale;  // scale * log2(e)
    float scale;
};

constexpr int kBwdThreads = 320;  // TMA warp, MMA warp, dS warpgroup, dQ warpgroup
// Query rows per block of the backward kernel: the height of the TMA boxes of
// its Q and dO maps (d = 128: 64-row blocks, so two blocks' scores fit in
// tensor memory; d = 64: 128).
constexpr int bwd_q_rows(int d) { return d == 128 ? 64 : 128; }

size_t bwd_workspace_bytes(int BH, int Nq, int d);
// sm_count: the persistent d = 128 kernel runs one CTA per SM (at most one per unit).
cudaError_t launch_bwd(int d, const BwdParams& p, int sm_count, cudaStream_t stream);

}  // namespace attn

#include "attn.h"

namespace attn {

// Device address of the calling device's status word (api.cu).
attn_status_t status_word_address(unsigned** out);

}  // namespace attn
