// decode.cu -- one-token attention over a paged KV cache, split over pages.
//
// "FlashAttention V3 实战: Hopper 架构下的 Paged KV Cache 协同优化",
// section 3.2: each request's keys live in fixed-size pages named by a block
// table (the vLLM / SGLang layout).  Decode is bound by HBM reads (the same
// page, opening paragraph: the bottleneck is the HBM access pattern), so the
// kernel streams every needed K/V byte exactly once with wide coalesced loads
// and keeps the arithmetic on the CUDA cores.
//
// Split kernel: CTA = (head group, split, request).  A split is a run of
// pages_per_split pages of one request.  A warp owns 32 / (d/8) heads; each
// lane holds 8 contiguous head dims of one head, so one 16-byte load per lane
// per token covers whole K (or V) rows of several heads, and the heads of a
// token are contiguous in memory ([page][slot][head][d]).  Scores are reduced
// across the d/8 lanes of a head with the xor-shuffle butterfly of "Capstone:
// CUDA Softmax 与 Attention 算子", section 3.3.  Tokens are processed in
// chunks of 8 with the online-softmax update of the same page, section 2.2
// (running max m, denominator l, rescale e^(m_old - m_new)), in log2 units.
// The split writes its unnormalised partial (O_s, m_s, l_s).
//
// Merge kernel: one warp per (request, head) combines the splits with the
// (m, l, O) merge of section 2.2 step 4:
//   m = max_s m_s,  l = sum_s l_s 2^(m_s - m),  O = sum_s 2^(m_s - m) O_s / l.
#include <cmath>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kChunk = 8;          // tokens per online-softmax update
constexpr int kSplitTokens = 128;  // target tokens per split

struct U4 {
    uint32_t x, y, z, w;
};

// 16-byte streaming load: read once, do not keep in L1.
__device__ __forceinline__ U4 ld_stream(const void* ptr) {
    U4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr));
    return r;
}

__device__ __forceinline__ float dot8(const float* q, const U4& k) {
    float a = q[0] * bf16lo_to_f32(k.x);
    a = fmaf(q[1], bf16hi_to_f32(k.x), a);
    a = fmaf(q[2], bf16lo_to_f32(k.y), a);
    a = fmaf(q[3], bf16hi_to_f32(k.y), a);
    a = fmaf(q[4], bf16lo_to_f32(k.z), a);
    a = fmaf(q[5], bf16hi_to_f32(k.z), a);
    a = fmaf(q[6], bf16lo_to_f32(k.w), a);
    a = fmaf(q[7], bf16hi_to_f32(k.w), a);
    return a;
}

__device__ __forceinline__ void axpy8(float* acc, float p, const U4& v) {
    acc[0] = fmaf(p, bf16lo_to_f32(v.x), acc[0]);
    acc[1] = fmaf(p, bf16hi_to_f32(v.x), acc[1]);
    acc[2] = fmaf(p, bf16lo_to_f32(v.y), acc[2]);
    acc[3] = fmaf(p, bf16hi_to_f32(v.y), acc[3]);
    acc[4] = fmaf(p, bf16lo_to_f32(v.z), acc[4]);
    acc[5] = fmaf(p, bf16hi_to_f32(v.z), acc[5]);
    acc[6] = fmaf(p, bf16lo_to_f32(v.w), acc[6]);
    acc[7] = fmaf(p, bf16hi_to_f32(v.w), acc[7]);
}

__device__ __forceinline__ int clamp_len(int len, int cap, unsigned* status) {
    if (len < 0 || len > cap) {
        atomicOr(status, 1u << kStatusDeviceData);
        return len < 0 ? 0 : cap;
    }
    return len;
}

template <int D>
__global__ void __launch_bounds__(512) decode_split_kernel(const DecodeParams p) {
    constexpr int LPH = D / 8;   // lanes per head
    constexpr int HPW = 32 / LPH;  // heads per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;
    const int r = blockIdx.z, split = blockIdx.y;
    const int head = (blockIdx.x * wpc + warp) * HPW + lane / LPH;
    const int sub = lane % LPH;  // which 8 dims of the head
    const bool active = head < p.H;

    const int cap = p.max_pages * p.page_size;
    const int len = clamp_len(__ldg(p.seq_lens + r), cap, p.status);
    const int t0 = split * p.pages_per_split * p.page_size;
    if (t0 >= len) return;  // this split is past the request's last page
    const int t1 = min(len, t0 + p.pages_per_split * p.page_size);

    float q[8];
    {
        U4 qq;
        qq.x = qq.y = qq.z = qq.w = 0u;
        if (active) qq = *reinterpret_cast<const U4*>(p.q + ((size_t)r * p.H + head) * D + sub * 8);
        q[0] = bf16lo_to_f32(qq.x); q[1] = bf16hi_to_f32(qq.x);
        q[2] = bf16lo_to_f32(qq.y); q[3] = bf16hi_to_f32(qq.y);
        q[4] = bf16lo_to_f32(qq.z); q[5] = bf16hi_to_f32(qq.z);
        q[6] = bf16lo_to_f32(qq.w); q[7] = bf16hi_to_f32(qq.w);
#pragma unroll
        for (int c = 0; c < 8; ++c) q[c] *= p.c_scale;
    }

    float m = -INFINITY, l = 0.f;
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;

    const size_t tok_stride = (size_t)p.H * D;  // elements between consecutive slots
    for (int t = t0; t < t1; t += kChunk) {
        const int page = __ldg(p.block_table + (size_t)r * p.max_pages + t / p.page_size);
        const bool page_ok = page >= 0 && page < p.num_pages;
        if (!page_ok) {
            if (lane == 0) atomicOr(p.status, 1u << kStatusDeviceData);
            continue;
        }
        const size_t base = ((size_t)page * p.page_size + (t % p.page_size)) * tok_stride + (size_t)head * D + sub * 8;
        U4 kr[kChunk], vr[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const bool ok = active && (t + i < t1);
            kr[i].x = kr[i].y = kr[i].z = kr[i].w = 0u;
            vr[i] = kr[i];
            if (ok) {
                kr[i] = ld_stream(p.k_cache + base + i * tok_stride);
                vr[i] = ld_stream(p.v_cache + base + i * tok_stride);
            }
        }
        float x[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) x[i] = dot8(q, kr[i]);
#pragma unroll
        for (int o = LPH / 2; o >= 1; o >>= 1) {
#pragma unroll
            for (int i = 0; i < kChunk; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], o);
        }
        float mc = -INFINITY;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            if (t + i >= t1) x[i] = -INFINITY;
            mc = fmaxf(mc, x[i]);
        }
        const float m_new = fmaxf(m, mc);
        const float alpha = ex2(m - m_new);  // m = -inf -> 0
        l *= alpha;
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] *= alpha;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const float pi = ex2(x[i] - m_new);
            l += pi;
            axpy8(acc, pi, vr[i]);
        }
        m = m_new;
    }

    if (!active) return;
    const size_t rec = ((size_t)r * p.H + head) * p.max_splits + split;
    float4* po = reinterpret_cast<float4*>(p.part_o + rec * D + sub * 8);
    po[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    po[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if (sub == 0) *reinterpret_cast<float2*>(p.part_ml + rec * 2) = make_float2(m, l);
}

template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p) {
    constexpr int PER = D / 32;  // output dims per lane
    const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= p.B * p.H) return;
    const int r = gw / p.H;
    const int cap = p.max_pages * p.page_size;
    const int len = clamp_len(__ldg(p.seq_lens + r), cap, p.status);
    const int n_pages = (len + p.page_size - 1) / p.page_size;
    const int ns = (n_pages + p.pages_per_split - 1) / p.pages_per_split;
    const size_t rec0 = (size_t)gw * p.max_splits;

    float m = -INFINITY;
    for (int s = lane; s < ns; s += 32) m = fmaxf(m, p.part_ml[(rec0 + s) * 2]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float l = 0.f;
    for (int s = lane; s < ns; s += 32) {
        const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + (rec0 + s) * 2);
        l += ml.y * ex2(ml.x - m);
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
cudaError_t launch_d(const DecodeParams& p, cudaStream_t stream) {
    constexpr int HPW = 32 / (D / 8);
    int warps = (p.H + HPW - 1) / HPW;
    if (warps > 16) warps = 16;
    const int groups = (p.H + warps * HPW - 1) / (warps * HPW);
    dim3 grid(groups, p.max_splits, p.B);
    decode_split_kernel<D><<<grid, warps * 32, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int total_warps = p.B * p.H;
    const int blocks = (total_warps + 7) / 8;
    decode_merge_kernel<D><<<blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

DecodePlan decode_plan(int B, int H, int d, int page_size, int max_pages) {
    DecodePlan pl{};
    int pps = kSplitTokens / page_size;
    if (pps < 1) pps = 1;
    pl.pages_per_split = pps;
    pl.max_splits = (max_pages + pps - 1) / pps;
    if (pl.max_splits < 1) pl.max_splits = 1;
    const size_t recs = (size_t)B * H * pl.max_splits;
    pl.part_o_bytes = recs * d * sizeof(float);
    pl.part_ml_bytes = recs * 2 * sizeof(float);
    const size_t align = 256;
    pl.workspace_bytes = (pl.part_o_bytes + align - 1) / align * align + pl.part_ml_bytes;
    return pl;
}

cudaError_t launch_paged_decode(int d, const DecodeParams& p, cudaStream_t stream) {
    if (d == 128) return launch_d<128>(p, stream);
    if (d == 64) return launch_d<64>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn

// ---------------------------------------------------------------- allocation-free variant
//
// attn_paged_decode_noalloc: the same split + merge kernels, with the
// split partials kept in a fixed device array of ATTN_NOALLOC_SCRATCH_BYTES
// that this file owns instead of a caller-provided workspace.  The array is
// part of the library image: every device that loads the library holds it
// until the process exits.  In host code its name is only a host-side
// stand-in, so its device address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels.

namespace attn {

static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxScratchDevices];

// Device address of the scratch array on the current device (first call per
// device resolves it; that first call should happen before any stream capture).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

// Split plan for the fixed scratch: the default number of pages per split,
// or the smallest coarser one whose partials fit in `cap` bytes.  Returns
// false when even one split per request does not fit.  Closed form: with
// bytes(s) = roundup(B*H*s*d*4, 256) + B*H*s*8 the partials of s splits per
// request, s_fit is the largest s with bytes(s) <= cap, and the smallest
// pages-per-split giving at most s_fit splits is ceil(max_pages / s_fit).
bool capped_plan(int B, int H, int d, int page_size, int max_pages, size_t cap, DecodePlan* out) {
    const size_t rec = (size_t)B * H;  // records per split index
    auto bytes = [&](size_t s) { return (rec * s * d * sizeof(float) + 255) / 256 * 256 + rec * s * 2 * sizeof(float); };
    size_t s_fit = cap / (rec * (d + 2) * sizeof(float));  // ignores the 256-byte round-up: at most one too many
    while (s_fit > 0 && bytes(s_fit) > cap) --s_fit;
    if (s_fit < 1) return false;
    int pps = 128 / page_size;
    if (pps < 1) pps = 1;
    const size_t need = ((size_t)max_pages + s_fit - 1) / s_fit;
    if (need > (size_t)pps) pps = (int)need;
    DecodePlan pl{};
    pl.pages_per_split = pps;
    pl.max_splits = (max_pages + pps - 1) / pps;
    pl.part_o_bytes = rec * pl.max_splits * d * sizeof(float);
    pl.part_ml_bytes = rec * pl.max_splits * 2 * sizeof(float);
    pl.workspace_bytes = (pl.part_o_bytes + 255) / 256 * 256 + pl.part_ml_bytes;
    if (pl.workspace_bytes > cap) return false;  // cannot happen: max_splits <= s_fit
    *out = pl;
    return true;
}

}  // namespace

}  // namespace attn

extern "C" attn_status_t attn_paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                   const int32_t* block_table, const int32_t* seq_lens, int B,
                                                   int H, int d, int page_size, int max_pages_per_seq,
                                                   int num_pages, float scale, void* o, float* lse,
                                                   void* stream) {
    using namespace attn;
    auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || max_pages_per_seq < 1 || num_pages < 1 || page_size < 1) return ATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(o)) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return ATTN_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || page_size < 8 || page_size > 1024 || page_size % 8 != 0)
        return ATTN_ERR_UNSUPPORTED;
    if ((long long)max_pages_per_seq * page_size > 0x7fffffffLL || (long long)B * max_pages_per_seq > 0x7fffffffLL)
        return ATTN_ERR_INVALID_ARG;
    DecodePlan pl{};
    if (!capped_plan(B, H, d, page_size, max_pages_per_seq, (size_t)ATTN_NOALLOC_SCRATCH_BYTES, &pl))
        return ATTN_ERR_WORKSPACE;  // the partials of even one split per request exceed the fixed scratch
    if (pl.max_splits > 65535 || B > 65535) return ATTN_ERR_UNSUPPORTED;

    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned* status = nullptr;
    attn_status_t st = status_word_address(&status);
    if (st != ATTN_OK) return st;

    DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.k_cache = static_cast<const uint16_t*>(k_cache);
    p.v_cache = static_cast<const uint16_t*>(v_cache);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.part_o = static_cast<float*>(scratch);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) + (pl.workspace_bytes - pl.part_ml_bytes));
    p.o = static_cast<uint16_t*>(o);
    p.lse = lse;
    p.status = status;
    p.B = B;
    p.H = H;
    p.page_size = page_size;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.pages_per_split = pl.pages_per_split;
    p.max_splits = pl.max_splits;
    p.c_scale = scale * 1.4426950408889634f;
    return launch_paged_decode(d, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
