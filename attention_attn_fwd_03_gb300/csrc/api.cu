// api.cu -- the extern "C" entry points declared in include/attn.h.
//
// Host-side only: argument validation (nothing is enqueued on a bad
// argument), TMA tensor-map encoding, per-device cached state (the device
// status word's address), the kernel launches, and the chunked copy/compute
// pipeline of attn_fwd_host (two streams and ten events per device, created
// on its first call).  No memory is allocated here or in any kernel.
#include <cmath>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "kernels.h"

namespace attn {

// Bit k set <=> a kernel reported status code k (ATTN_ERR_TIMEOUT,
// ATTN_ERR_DEVICE_DATA).  One word per device; cleared by attn_device_status.
__device__ unsigned g_status_word;
// The word as attn_device_status last took it (read and cleared in one atomic
// step, so a bit set by a kernel on another stream meanwhile is never lost).
__device__ unsigned g_status_taken;

namespace {
__global__ void status_take_kernel() { g_status_taken = atomicExch(&g_status_word, 0u); }
std::mutex g_take_mu;  // one take at a time per process (g_status_taken is shared)
}  // namespace

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    unsigned* status = nullptr;
    int sm_count = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

attn_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Per-device set-up, once: the status word's device address.
attn_status_t device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return ATTN_ERR_CUDA;
        s.status = static_cast<unsigned*>(ptr);
        if (cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            s.sm_count < 1)
            return ATTN_ERR_CUDA;
        s.ready = true;
    }
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return ATTN_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = &s;
    return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D map over a [BH, rows, d] tensor.  Operand maps: box = (128 bytes of d,
// box_rows rows (128 unless given), 1) with 128-byte swizzle; output map:
// box = (32 elements, 32 rows, 1), no swizzle.  Zero fill outside the tensor;
// stores are clipped.
bool make_map(CUtensorMap* map, const void* base, bool fp8, int d, long long rows, long long bh, bool out,
              int box_rows = 128) {
    const int eb = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)bh};
    cuuint64_t strides[2] = {(cuuint64_t)d * eb, (cuuint64_t)rows * d * eb};
    cuuint32_t box[3] = {out ? 32u : (cuuint32_t)(128 / eb), out ? 32u : (cuuint32_t)box_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          out ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The decoupled prefill kernel (prefill_sp.cu) is the faster one when a
// unit -- two 128-row query tiles -- streams many KV blocks; with short rows
// its unit boundaries, where both tiles end together, cost more than its
// overlap gains, and the turn-based kernel (prefill.cu) is faster.  Measured
// on GB300 (bf16 d = 128): 16 blocks per unit (4x16x2048, non-causal) favour
// the turn-based kernel by 12%; 64 (FP8 2x16x8192) and ~128 (causal
// 1x32x32768) favour the decoupled one by 4% and 7%.
constexpr double kSpMinMeanBlocks = 48.0;

// Mean number of KV blocks a unit streams (the longer of its two tiles).
double mean_unit_blocks(int Nq, int Nk, int causal) {
    const long long kv_blocks = ((long long)Nk + 127) / 128;
    if (!causal) return (double)kv_blocks;
    const long long pairs = ((long long)Nq + 255) / 256;
    auto tile = [&](long long q0) -> long long {  // blocks of tile [q0, q0 + 128) clipped to Nq
        if (q0 >= Nq) return 0;
        const long long rows = (Nq - q0) < 128 ? (Nq - q0) : 128;
        const long long last_key = q0 + rows - 1 + (Nk - Nq);
        if (last_key < 0) return 0;
        const long long nb = last_key / 128 + 1;
        return nb < kv_blocks ? nb : kv_blocks;
    };
    // J of pair i grows with i; sum it exactly for up to 2^16 pairs, else
    // take 4096 evenly spaced pairs
    const long long step = pairs <= 65536 ? 1 : pairs / 4096;
    double sum = 0.0;
    long long n = 0;
    for (long long i = 0; i < pairs; i += step, ++n) {
        const long long a = tile(2 * i * 128), b = tile((2 * i + 1) * 128);
        sum += (double)(a > b ? a : b);
    }
    return n ? sum / (double)n : 0.0;
}

attn_status_t prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                      int Nk, int d, float scale, int causal, bool fp8, float dq, float dk, float dv,
                      void* stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (fp8 && !(std::isfinite(dq) && dq > 0.f && std::isfinite(dk) && dk > 0.f && std::isfinite(dv) && dv > 0.f))
        return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
    if (fp8 ? d != 128 : (d != 64 && d != 128)) return ATTN_ERR_UNSUPPORTED;

    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;

    const long long BH = (long long)B * H;
    PrefillParams p;
    std::memset(&p, 0, sizeof p);
    if (!make_map(&p.tm_q, q, fp8, d, Nq, BH, false) || !make_map(&p.tm_k, k, fp8, d, Nk, BH, false) ||
        !make_map(&p.tm_v, v, fp8, d, Nk, BH, false) || !make_map(&p.tm_o, o, false, d, Nq, BH, true))
        return ATTN_ERR_CUDA;
    p.lse = lse;
    p.o = static_cast<uint16_t*>(o);
    p.status = ds->status;
    p.BH = (int)BH;
    p.Nq = Nq;
    p.Nk = Nk;
    p.causal = causal;
    p.n_pairs = (Nq + 255) / 256;
    const float log2e = 1.4426950408889634f;
    p.c_scale = fp8 ? scale * dq * dk * log2e : scale * log2e;
    p.o_scale = fp8 ? dv : 1.f;
    const long long units = (long long)p.n_pairs * BH;
    if (units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    p.n_units = (int)units;
    const int grid = units < ds->sm_count ? (int)units : ds->sm_count;  // persistent: one CTA per SM
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (mean_unit_blocks(Nq, Nk, causal) >= kSpMinMeanBlocks) return from_cuda(launch_prefill_sp(d, fp8, p, grid, s));
    return from_cuda(launch_prefill(d, fp8, p, grid, s));
}

bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

// Checks shared by the paged size query and the paged call; returns ATTN_OK
// or the status to report.
attn_status_t paged_sizes_ok(int B, int total_q, int max_q_len, int H, int H_kv, int d, int page_size,
                             int max_pages) {
    if (B < 1 || total_q < 1 || max_q_len < 1 || max_q_len > total_q || H < 1 || H_kv < 1 || max_pages < 1)
        return ATTN_ERR_INVALID_ARG;
    if (H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
    if (H / H_kv > 128 || (d != 64 && d != 128) || !pow2_in(page_size, 8, 1024)) return ATTN_ERR_UNSUPPORTED;
    if ((long long)max_pages * page_size > 0x7fffffffLL || (long long)B * max_pages > 0x7fffffffLL ||
        (long long)total_q * H > 0x7fffffffLL)
        return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

// Q map over [total_q, H, d]: box (64 elements, G heads, T tokens).  Cache
// map over [slots, H_kv, d]: box (64 elements, 1 head, R rows).  Both with
// 128-byte swizzle and zero fill outside the tensor.
bool make_paged_map(CUtensorMap* map, const void* base, int d, long long heads, long long rows, int box_heads,
                    int box_rows) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---- ragged prefill: the prefill kernel over variable-length sequences.
//
// Launches whose sequences bring at least kRaggedMinQ query tokens run on
// the prefill kernel in its ragged mode (two 128-row tiles of one query
// head per unit, the keys of its KV head streamed once for both); shorter
// ones -- decode steps, short chunks -- on the paged kernel, which packs the
// G query heads of a KV head into one tile.
constexpr int kRaggedMinQ = 128;

bool use_ragged(int max_q_len) { return max_q_len >= kRaggedMinQ; }

// Maps of the ragged mode over a token-major [rows, heads, d] tensor: dims
// (d, rows, heads), so that a box walks rows of one head.  Operand maps: box
// (64 elements, box_rows rows, 1 head), 128-byte swizzle; output map: box (32
// elements, 32 rows, 1 head), no swizzle.  Zero fill outside the tensor;
// stores are clipped.
bool make_rows_map(CUtensorMap* map, const void* base, int d, long long heads, long long rows, int box_rows,
                   bool out) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)heads * d * 2, (cuuint64_t)d * 2};
    cuuint32_t box[3] = {out ? 32u : 64u, out ? 32u : (cuuint32_t)box_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          out ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Keys: paged (block_table non-null: rows = num_pages * page_size slots,
// R = min(page_size, 128) rows per box) or contiguous (rows = total_k, R = 128).
attn_status_t ragged_prefill(DeviceState* ds, const void* q, const void* k, const void* v,
                             const int32_t* block_table, const int32_t* cu_q, const int32_t* seq_lens,
                             const int32_t* cu_k, int B, int total_q, int max_q_len, int H, int H_kv, int d,
                             int page_size, int max_pages, int num_pages, long long kv_rows, int kv_cap, float scale,
                             int causal, void* o, float* lse, void* workspace, cudaStream_t stream) {
    PrefillParams p;
    std::memset(&p, 0, sizeof p);
    const int R = block_table ? (page_size < 128 ? page_size : 128) : 128;
    if (!make_rows_map(&p.tm_q, q, d, H, total_q, 128, false) || !make_rows_map(&p.tm_k, k, d, H_kv, kv_rows, R, false) ||
        !make_rows_map(&p.tm_v, v, d, H_kv, kv_rows, R, false) || !make_rows_map(&p.tm_o, o, d, H, total_q, 0, true))
        return ATTN_ERR_CUDA;
    int* n_listed = static_cast<int*>(workspace);
    int4* units = reinterpret_cast<int4*>(static_cast<char*>(workspace) + 256);
    p.lse = lse;
    p.status = ds->status;
    p.causal = causal;
    p.c_scale = scale * 1.4426950408889634f;
    p.o_scale = 1.f;
    p.units = units;
    p.n_listed = n_listed;
    p.block_table = block_table;
    p.o = static_cast<uint16_t*>(o);
    p.H = H;
    p.G = H / H_kv;
    p.page_size = page_size;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.rows_per_box = R;
    p.kv_rows = (int)kv_rows;
    RaggedSched sp;
    std::memset(&sp, 0, sizeof sp);
    sp.cu_q = cu_q;
    sp.seq_lens = block_table ? seq_lens : nullptr;
    sp.cu_k = block_table ? nullptr : cu_k;
    sp.units = units;
    sp.n_listed = n_listed;
    sp.status = ds->status;
    sp.B = B;
    sp.H = H;
    sp.total_q = total_q;
    sp.max_q_len = max_q_len;
    sp.kv_cap = kv_cap;
    sp.causal = causal;
    sp.kv_bytes_per_key = H_kv * d * 4;
    const long long upper = (long long)B * ((max_q_len + 255) / 256) * H;  // units the list can hold
    const int grid = upper < ds->sm_count ? (int)upper : ds->sm_count;     // persistent: one CTA per SM
    return from_cuda(launch_ragged_prefill(d, sp, p, grid, stream));
}

// ---- host-staged prefill: copy in, compute, copy out, chunk by chunk.
//
// The (b, h) range is cut into chunks.  Chunk c uses workspace slot
// c % kHostSlots: its Q/K/V are copied in on stream s_in, its kernels run on
// the caller's stream, its O/LSE are copied out on stream s_out.  Events per
// slot order the three stages and the reuse of a slot three chunks later:
//   copy-in of c    after the kernels of c - kHostSlots (comp_done)
//   kernels of c    after copy-in of c (in_done) and copy-out of c - kHostSlots (out_done)
//   copy-out of c   after the kernels of c (comp_done)
constexpr int kHostSlots = 3;
constexpr int kHostMaxModes = 8;

struct HostStage {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t entry = nullptr;
    cudaEvent_t in_done[kHostSlots] = {}, comp_done[kHostSlots] = {}, out_done[kHostSlots] = {};
};

std::mutex g_host_mu;
HostStage g_host[kMaxDevices];

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Byte sizes of the buffers in one slot (each rounded up to 256 bytes).
struct SlotLayout {
    size_t q, kv, o, lse, per_mode, slot;
};

SlotLayout slot_layout(long long cb, int Nq, int Nk, int d, int n_modes) {
    SlotLayout L;
    L.q = round_up256((size_t)cb * Nq * d * 2);
    L.kv = round_up256((size_t)cb * Nk * d * 2);
    L.o = L.q;
    L.lse = round_up256((size_t)cb * Nq * 4);
    L.per_mode = L.o + L.lse;
    L.slot = L.q + 2 * L.kv + (size_t)n_modes * L.per_mode;
    return L;
}

// Pairs per chunk: the caller's, else about an eighth of B*H.
long long host_chunk(long long BH, int chunk_bh) {
    long long cb = chunk_bh > 0 ? chunk_bh : (BH + 7) / 8;
    return cb < BH ? cb : BH;
}

// Sizes accepted by the host-staged call; the slot arithmetic stays far
// from size_t overflow.
bool host_sizes_ok(int B, int H, int Nq, int Nk, int d, int n_modes, int chunk_bh) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || n_modes < 1 || n_modes > kHostMaxModes) return false;
    if (d != 64 && d != 128) return false;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return false;
    const double cb = (double)host_chunk(BH, chunk_bh);
    const double slot = cb * (3.0 * Nq + 2.0 * Nk) * d * 2.0 * (n_modes + 2) + 1e6;
    return slot * kHostSlots < 1e18;
}

// Host (page-locked, pageable or managed) memory, i.e. not device memory.
bool host_memory(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type != cudaMemoryTypeDevice;
}

bool device_memory(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

attn_status_t host_stage_state(HostStage** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    HostStage& h = g_host[dev];
    if (!h.ready) {
        if (cudaStreamCreateWithFlags(&h.s_in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&h.s_out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&h.entry, cudaEventDisableTiming) != cudaSuccess)
            return ATTN_ERR_CUDA;
        for (int s = 0; s < kHostSlots; ++s)
            if (cudaEventCreateWithFlags(&h.in_done[s], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&h.comp_done[s], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&h.out_done[s], cudaEventDisableTiming) != cudaSuccess)
                return ATTN_ERR_CUDA;
        h.ready = true;
    }
    *out = &h;
    return ATTN_OK;
}

}  // namespace

// Device address of the calling device's status word (set-up on first use).
attn_status_t status_word_address(unsigned** out) {
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    *out = ds->status;
    return ATTN_OK;
}

}  // namespace attn

using namespace attn;

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                       int Nk, int d, float scale, int causal, void* stream) {
    return prefill(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, false, 1.f, 1.f, 1.f, stream);
}

attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v8, float q_descale, float k_descale,
                           float v_descale, void* o, float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                           int causal, void* stream) {
    return prefill(q8, k8, v8, o, lse, B, H, Nq, Nk, d, scale, causal, true, q_descale, k_descale, v_descale,
                   stream);
}

size_t attn_paged_decode_workspace_size(int B, int H, int d, int max_pages_per_seq, int page_size) {
    if (B < 1 || H < 1 || (d != 64 && d != 128) || page_size < 8 || page_size > 1024 || page_size % 8 != 0 ||
        max_pages_per_seq < 1)
        return 0;
    return decode_plan(B, H, d, page_size, max_pages_per_seq).workspace_bytes;
}

attn_status_t attn_paged_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                const int32_t* seq_lens, int B, int H, int d, int page_size, int max_pages_per_seq,
                                int num_pages, float scale, void* o, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || max_pages_per_seq < 1 || num_pages < 1 || page_size < 1) return ATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return ATTN_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || page_size < 8 || page_size > 1024 || page_size % 8 != 0)
        return ATTN_ERR_UNSUPPORTED;
    if ((long long)max_pages_per_seq * page_size > 0x7fffffffLL || (long long)B * max_pages_per_seq > 0x7fffffffLL)
        return ATTN_ERR_INVALID_ARG;
    const DecodePlan pl = decode_plan(B, H, d, page_size, max_pages_per_seq);
    if (!workspace || workspace_bytes < pl.workspace_bytes || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    if (pl.max_splits > 65535 || B > 65535) return ATTN_ERR_UNSUPPORTED;

    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;

    DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.q = static_cast<const uint16_t*>(q);
    p.k_cache = static_cast<const uint16_t*>(k_cache);
    p.v_cache = static_cast<const uint16_t*>(v_cache);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.part_o = static_cast<float*>(workspace);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + (pl.workspace_bytes - pl.part_ml_bytes));
    p.o = static_cast<uint16_t*>(o);
    p.lse = lse;
    p.status = ds->status;
    p.B = B;
    p.H = H;
    p.page_size = page_size;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.pages_per_split = pl.pages_per_split;
    p.max_splits = pl.max_splits;
    p.c_scale = scale * 1.4426950408889634f;
    return from_cuda(launch_paged_decode(d, p, static_cast<cudaStream_t>(stream)));
}

size_t attn_paged_fwd_workspace_size(int B, int total_q, int max_q_len, int H, int H_kv, int d, int page_size,
                                     int max_pages_per_seq) {
    if (paged_sizes_ok(B, total_q, max_q_len, H, H_kv, d, page_size, max_pages_per_seq) != ATTN_OK) return 0;
    if (use_ragged(max_q_len)) return ragged_workspace_bytes(B, max_q_len, H);
    return paged_plan(total_q, max_q_len, B, H, H_kv, d, page_size, max_pages_per_seq).workspace_bytes;
}

attn_status_t attn_paged_fwd(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                             const int32_t* cu_seqlens_q, const int32_t* seq_lens, int B, int total_q,
                             int max_q_len, int H, int H_kv, int d, int page_size, int max_pages_per_seq,
                             int num_pages, float scale, int causal, void* o, float* lse, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o) return ATTN_ERR_INVALID_ARG;
    if (!cu_seqlens_q && (total_q != B || max_q_len != 1)) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = paged_sizes_ok(B, total_q, max_q_len, H, H_kv, d, page_size, max_pages_per_seq);
    if (st != ATTN_OK) return st;
    if (num_pages < 1 || (long long)num_pages * page_size > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    auto a4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
    if (!a4(block_table) || !a4(seq_lens) || (cu_seqlens_q && !a4(cu_seqlens_q)) || (lse && !a4(lse)))
        return ATTN_ERR_INVALID_ARG;
    if (use_ragged(max_q_len)) {
        const size_t need = ragged_workspace_bytes(B, max_q_len, H);
        if ((long long)B * ((max_q_len + 255) / 256) * H > 0x3fffffffLL) return ATTN_ERR_INVALID_ARG;
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
        DeviceState* ds = nullptr;
        st = device_state(&ds);
        if (st != ATTN_OK) return st;
        return ragged_prefill(ds, q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, nullptr, B, total_q,
                              max_q_len, H, H_kv, d, page_size, max_pages_per_seq, num_pages,
                              (long long)num_pages * page_size, max_pages_per_seq * page_size, scale, causal, o, lse,
                              workspace, static_cast<cudaStream_t>(stream));
    }
    const PagedPlan pl = paged_plan(total_q, max_q_len, B, H, H_kv, d, page_size, max_pages_per_seq);
    if (pl.n_units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pl.workspace_bytes || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;

    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != ATTN_OK) return st;

    PagedParams p;
    std::memset(&p, 0, sizeof p);
    const long long slots = (long long)num_pages * page_size;
    const int R = page_size < 128 ? page_size : 128;
    if (!make_paged_map(&p.tm_q, q, d, H, total_q, pl.G, pl.T) ||
        !make_paged_map(&p.tm_k, k_cache, d, H_kv, slots, 1, R) ||
        !make_paged_map(&p.tm_v, v_cache, d, H_kv, slots, 1, R))
        return ATTN_ERR_CUDA;
    p.block_table = block_table;
    p.cu_q = cu_seqlens_q;
    p.seq_lens = seq_lens;
    p.o = static_cast<uint16_t*>(o);
    p.lse = lse;
    p.sched = static_cast<int*>(workspace);
    char* ws = static_cast<char*>(workspace);
    p.sched_list = reinterpret_cast<int4*>(ws + pl.list_offset);
    if (pl.n_splits > 1) {
        p.part_o = reinterpret_cast<float*>(ws + pl.part_o_offset);
        p.part_ml = reinterpret_cast<float*>(ws + pl.part_ml_offset);
        if (pl.whole_offset != 0) p.whole = reinterpret_cast<int*>(ws + pl.whole_offset);
    }
    p.status = ds->status;
    p.B = B;
    p.H = H;
    p.H_kv = H_kv;
    p.G = pl.G;
    p.T = pl.T;
    p.total_q = total_q;
    p.max_q_len = max_q_len;
    p.n_qt = pl.n_qt;
    p.page_size = page_size;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.rows_per_box = R;
    p.kv_rows = (int)slots;
    p.causal = causal;
    p.n_splits = pl.n_splits;
    p.split_blocks = pl.split_blocks;
    p.n_units = (int)pl.n_units;
    p.q_tile_bytes = (uint32_t)(d / 64) * (uint32_t)(pl.G * pl.T) * 128u;
    p.c_scale = scale * 1.4426950408889634f;
    const int grid = pl.n_units < ds->sm_count ? (int)pl.n_units : ds->sm_count;  // persistent: one CTA per SM
    p.n_ctas = grid;
    return from_cuda(launch_paged(d, p, grid, static_cast<cudaStream_t>(stream)));
}

size_t attn_varlen_fwd_workspace_size(int B, int total_q, int max_q_len, int max_k_len, int H, int H_kv, int d) {
    if (max_k_len < 1) return 0;
    const int max_blocks = (int)(((long long)max_k_len + 127) / 128);
    if (paged_sizes_ok(B, total_q, max_q_len, H, H_kv, d, 128, max_blocks) != ATTN_OK) return 0;
    if (use_ragged(max_q_len)) return ragged_workspace_bytes(B, max_q_len, H);
    return paged_plan(total_q, max_q_len, B, H, H_kv, d, 128, max_blocks).workspace_bytes;
}

attn_status_t attn_varlen_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, int B, int total_q, int total_k, int max_q_len,
                              int max_k_len, int H, int H_kv, int d, float scale, int causal, void* o, float* lse,
                              void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !o) return ATTN_ERR_INVALID_ARG;
    if (total_k < 1 || max_k_len < 1 || max_k_len > total_k) return ATTN_ERR_INVALID_ARG;
    const int max_blocks = (int)(((long long)max_k_len + 127) / 128);
    attn_status_t st = paged_sizes_ok(B, total_q, max_q_len, H, H_kv, d, 128, max_blocks);
    if (st != ATTN_OK) return st;
    if ((long long)total_k + 128 > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    auto a4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
    if (!a4(cu_seqlens_q) || !a4(cu_seqlens_k) || (lse && !a4(lse))) return ATTN_ERR_INVALID_ARG;
    if (use_ragged(max_q_len)) {
        const size_t need = ragged_workspace_bytes(B, max_q_len, H);
        if ((long long)B * ((max_q_len + 255) / 256) * H > 0x3fffffffLL) return ATTN_ERR_INVALID_ARG;
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
        DeviceState* ds = nullptr;
        st = device_state(&ds);
        if (st != ATTN_OK) return st;
        return ragged_prefill(ds, q, k, v, nullptr, cu_seqlens_q, nullptr, cu_seqlens_k, B, total_q, max_q_len, H,
                              H_kv, d, 128, max_blocks, 0, total_k, total_k, scale, causal, o, lse, workspace,
                              static_cast<cudaStream_t>(stream));
    }
    const PagedPlan pl = paged_plan(total_q, max_q_len, B, H, H_kv, d, 128, max_blocks);
    if (pl.n_units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pl.workspace_bytes || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;

    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != ATTN_OK) return st;

    PagedParams p;
    std::memset(&p, 0, sizeof p);
    if (!make_paged_map(&p.tm_q, q, d, H, total_q, pl.G, pl.T) || !make_paged_map(&p.tm_k, k, d, H_kv, total_k, 1, 128) ||
        !make_paged_map(&p.tm_v, v, d, H_kv, total_k, 1, 128))
        return ATTN_ERR_CUDA;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.o = static_cast<uint16_t*>(o);
    p.lse = lse;
    p.sched = static_cast<int*>(workspace);
    char* ws = static_cast<char*>(workspace);
    p.sched_list = reinterpret_cast<int4*>(ws + pl.list_offset);
    if (pl.n_splits > 1) {
        p.part_o = reinterpret_cast<float*>(ws + pl.part_o_offset);
        p.part_ml = reinterpret_cast<float*>(ws + pl.part_ml_offset);
        if (pl.whole_offset != 0) p.whole = reinterpret_cast<int*>(ws + pl.whole_offset);
    }
    p.status = ds->status;
    p.B = B;
    p.H = H;
    p.H_kv = H_kv;
    p.G = pl.G;
    p.T = pl.T;
    p.total_q = total_q;
    p.max_q_len = max_q_len;
    p.n_qt = pl.n_qt;
    p.page_size = 128;
    p.max_pages = max_blocks;
    p.num_pages = 0;
    p.rows_per_box = 128;
    p.kv_rows = total_k;
    p.causal = causal;
    p.n_splits = pl.n_splits;
    p.split_blocks = pl.split_blocks;
    p.n_units = (int)pl.n_units;
    p.q_tile_bytes = (uint32_t)(d / 64) * (uint32_t)(pl.G * pl.T) * 128u;
    p.c_scale = scale * 1.4426950408889634f;
    const int grid = pl.n_units < ds->sm_count ? (int)pl.n_units : ds->sm_count;  // persistent: one CTA per SM
    p.n_ctas = grid;
    return from_cuda(launch_paged(d, p, grid, static_cast<cudaStream_t>(stream)));
}

size_t attn_bwd_workspace_size(int B, int H, int Nq, int d) {
    if (B < 1 || H < 1 || Nq < 1 || (d != 64 && d != 128) || (long long)B * H > 65535) return 0;
    return bwd_workspace_bytes(B * H, Nq, d);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                       float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return ATTN_ERR_UNSUPPORTED;  // grid.y holds batch * heads
    // the d = 128 kernel counts (batch*head, 128-key block) units in 32 bits
    if ((long long)B * H * (((long long)Nk + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv))
        return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    const int BH = B * H;
    const size_t need = bwd_workspace_bytes(BH, Nq, d);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;

    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;

    BwdParams p;
    std::memset(&p, 0, sizeof p);
    const int qrows = bwd_q_rows(d);  // query block height of the backward kernel
    if (!make_map(&p.tm_q, q, false, d, Nq, BH, false, qrows) || !make_map(&p.tm_k, k, false, d, Nk, BH, false) ||
        !make_map(&p.tm_v, v, false, d, Nk, BH, false) || !make_map(&p.tm_do, dout, false, d, Nq, BH, false, qrows))
        return ATTN_ERR_CUDA;
    const int nq_pad = (Nq + 127) / 128 * 128;
    char* ws = static_cast<char*>(workspace);
    p.dq_acc = reinterpret_cast<float*>(ws);
    {  // reduce target of the dQ boxes: 32 fp32 columns x 32 rows, 128-byte swizzle
        cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)nq_pad, (cuuint64_t)BH};
        cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)nq_pad * d * 4};
        cuuint32_t box[3] = {32u, 32u, 1u};
        cuuint32_t estr[3] = {1u, 1u, 1u};
        if (g_encode(&p.tm_dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.dq_acc, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return ATTN_ERR_CUDA;
    }
    p.lse2 = reinterpret_cast<float*>(ws + (size_t)BH * nq_pad * d * sizeof(float));
    p.dvec = p.lse2 + (size_t)BH * nq_pad;
    p.o = static_cast<const uint16_t*>(o);
    p.dout = static_cast<const uint16_t*>(dout);
    p.lse = lse;
    p.dq = static_cast<uint16_t*>(dq);
    p.dk = static_cast<uint16_t*>(dk);
    p.dv = static_cast<uint16_t*>(dv);
    p.status = ds->status;
    p.BH = BH;
    p.Nq = Nq;
    p.Nk = Nk;
    p.causal = causal;
    p.n_qblocks = nq_pad / 128;
    p.n_kblocks = (Nk + 127) / 128;
    p.nq_pad = nq_pad;
    p.c_scale = scale * 1.4426950408889634f;
    p.scale = scale;
    return from_cuda(launch_bwd(d, p, ds->sm_count, static_cast<cudaStream_t>(stream)));
}

size_t attn_fwd_host_workspace_size(int B, int H, int Nq, int Nk, int d, int n_modes, int chunk_bh) {
    if (!host_sizes_ok(B, H, Nq, Nk, d, n_modes, chunk_bh)) return 0;
    const long long cb = host_chunk((long long)B * H, chunk_bh);
    return (size_t)kHostSlots * slot_layout(cb, Nq, Nk, d, n_modes).slot;
}

attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, int n_modes, const int* causal,
                            void* const* o, float* const* lse, int B, int H, int Nq, int Nk, int d, float scale,
                            int chunk_bh, void* workspace, size_t workspace_bytes, void* stream) {
    // ---- validation: nothing is enqueued on a bad argument
    if (!q || !k || !v || !causal || !o) return ATTN_ERR_INVALID_ARG;
    if (n_modes < 1 || n_modes > kHostMaxModes) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (long long)B * H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    for (int m = 0; m < n_modes; ++m)
        if (!o[m] || (causal[m] != 0 && causal[m] != 1)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (!host_sizes_ok(B, H, Nq, Nk, d, n_modes, chunk_bh)) return ATTN_ERR_INVALID_ARG;
    const size_t need = attn_fwd_host_workspace_size(B, H, Nq, Nk, d, n_modes, chunk_bh);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_WORKSPACE;

    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    if (!host_memory(q) || !host_memory(k) || !host_memory(v)) return ATTN_ERR_INVALID_ARG;
    for (int m = 0; m < n_modes; ++m)
        if (!host_memory(o[m]) || (lse && lse[m] && !host_memory(lse[m]))) return ATTN_ERR_INVALID_ARG;
    if (!device_memory(workspace)) return ATTN_ERR_WORKSPACE;

    std::lock_guard<std::mutex> lock(g_host_mu);
    HostStage* hs = nullptr;
    st = host_stage_state(&hs);
    if (st != ATTN_OK) return st;

    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const long long BH = (long long)B * H;
    const long long cb = host_chunk(BH, chunk_bh);
    const long long n_chunks = (BH + cb - 1) / cb;
    const SlotLayout L = slot_layout(cb, Nq, Nk, d, n_modes);
    const size_t q_bh = (size_t)Nq * d * 2, kv_bh = (size_t)Nk * d * 2, l_bh = (size_t)Nq * 4;
    const uint8_t* hq = static_cast<const uint8_t*>(q);
    const uint8_t* hk = static_cast<const uint8_t*>(k);
    const uint8_t* hv = static_cast<const uint8_t*>(v);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
#define ATTN_CK(x)                                  \
    do {                                            \
        if ((x) != cudaSuccess) return ATTN_ERR_CUDA; \
    } while (0)

    // both copy streams start after the work already on the caller's stream
    ATTN_CK(cudaEventRecord(hs->entry, cs));
    ATTN_CK(cudaStreamWaitEvent(hs->s_in, hs->entry, 0));
    ATTN_CK(cudaStreamWaitEvent(hs->s_out, hs->entry, 0));
    for (long long c = 0; c < n_chunks; ++c) {
        const int slot = (int)(c % kHostSlots);
        const long long bh0 = c * cb;
        const long long n = (BH - bh0) < cb ? (BH - bh0) : cb;
        uint8_t* dq = ws + (size_t)slot * L.slot;
        uint8_t* dk = dq + L.q;
        uint8_t* dv = dk + L.kv;
        uint8_t* dout0 = dv + L.kv;
        // copy in
        if (c >= kHostSlots) ATTN_CK(cudaStreamWaitEvent(hs->s_in, hs->comp_done[slot], 0));
        ATTN_CK(cudaMemcpyAsync(dq, hq + bh0 * q_bh, n * q_bh, cudaMemcpyHostToDevice, hs->s_in));
        ATTN_CK(cudaMemcpyAsync(dk, hk + bh0 * kv_bh, n * kv_bh, cudaMemcpyHostToDevice, hs->s_in));
        ATTN_CK(cudaMemcpyAsync(dv, hv + bh0 * kv_bh, n * kv_bh, cudaMemcpyHostToDevice, hs->s_in));
        ATTN_CK(cudaEventRecord(hs->in_done[slot], hs->s_in));
        // compute: the chunk's n pairs as one [1, n] batch, one launch per mode
        ATTN_CK(cudaStreamWaitEvent(cs, hs->in_done[slot], 0));
        if (c >= kHostSlots) ATTN_CK(cudaStreamWaitEvent(cs, hs->out_done[slot], 0));
        for (int m = 0; m < n_modes; ++m) {
            uint8_t* dom = dout0 + (size_t)m * L.per_mode;
            float* dlm = (lse && lse[m]) ? reinterpret_cast<float*>(dom + L.o) : nullptr;
            st = prefill(dq, dk, dv, dom, dlm, 1, (int)n, Nq, Nk, d, scale, causal[m], false, 1.f, 1.f, 1.f, cs);
            if (st != ATTN_OK) return st;
        }
        ATTN_CK(cudaEventRecord(hs->comp_done[slot], cs));
        // copy out
        ATTN_CK(cudaStreamWaitEvent(hs->s_out, hs->comp_done[slot], 0));
        for (int m = 0; m < n_modes; ++m) {
            uint8_t* dom = dout0 + (size_t)m * L.per_mode;
            ATTN_CK(cudaMemcpyAsync(static_cast<uint8_t*>(o[m]) + bh0 * q_bh, dom, n * q_bh, cudaMemcpyDeviceToHost,
                                    hs->s_out));
            if (lse && lse[m])
                ATTN_CK(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse[m]) + bh0 * l_bh, dom + L.o, n * l_bh,
                                        cudaMemcpyDeviceToHost, hs->s_out));
        }
        ATTN_CK(cudaEventRecord(hs->out_done[slot], hs->s_out));
    }
    // later work on the caller's stream starts after the last copy out (the
    // copy-out stream runs in order, so that covers every chunk)
    ATTN_CK(cudaStreamWaitEvent(cs, hs->out_done[(n_chunks - 1) % kHostSlots], 0));
#undef ATTN_CK
    return ATTN_OK;
}

attn_status_t attn_selftest_wait_timeout(void* stream) {
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    return from_cuda(launch_selftest_timeout(ds->status, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_selftest_mma_rate(unsigned long long* cycles, int n_ctas, int n_groups, void* stream) {
    if (cycles == nullptr || (reinterpret_cast<uintptr_t>(cycles) & 7u) || n_ctas < 1 || n_ctas > 65535 ||
        n_groups < 1 || n_groups > (1 << 20))
        return ATTN_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    return from_cuda(launch_selftest_mma_rate(n_ctas, n_groups, cycles, ds->status, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_device_status(void* stream) {
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned word = 0;
    {
        std::lock_guard<std::mutex> lock(g_take_mu);
        status_take_kernel<<<1, 1, 0, s>>>();
        if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
        if (cudaMemcpyFromSymbolAsync(&word, g_status_taken, sizeof word, 0, cudaMemcpyDeviceToHost, s) !=
                cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    if (word & (1u << ATTN_ERR_TIMEOUT)) return ATTN_ERR_TIMEOUT;
    if (word & (1u << ATTN_ERR_DEVICE_DATA)) return ATTN_ERR_DEVICE_DATA;
    return ATTN_OK;
}

const char* attn_status_string(attn_status_t s) {
    switch (s) {
    case ATTN_OK: return "success";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA runtime or launch failure";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
    case ATTN_ERR_DEVICE_DATA: return "device-side length or page id out of range";
    }
    return "unknown status";
}

}  // extern "C"
