/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * Every forward entry point computes exact scaled-dot-product attention
 *     O = softmax(scale * Q K^T) V
 * ("FlashAttention V3 实战: Hopper 架构下的 Paged KV Cache 协同优化",
 * section 一, the attention formula; "Capstone: CUDA Softmax 与 Attention
 * 算子", section 1.1) in one tiled pass with the online-softmax running max m
 * and denominator l (same Capstone page, section 2.2 steps 3-5, and section
 * 4.1-4.2 for the loop order and the single final division), so the score
 * and probability matrices never reach device memory.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, except
 *     the tensors of attn_fwd_host, which live in host memory.  The
 *     library allocates no memory and frees nothing; it keeps only
 *     per-device cached kernel attributes, one device status word (see
 *     attn_device_status) and, once attn_fwd_host has run on a device, that
 *     call's two streams and ten events.
 *   - Layouts are dense row-major ("BHSD"): element (b, h, i, c) of a
 *     [B, H, N, d] tensor is at ((b*H + h)*N + i)*d + c.
 *   - Every device pointer must be 16-byte aligned (host pointers of
 *     attn_fwd_host need no alignment).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous: they validate their arguments on the
 *     host, enqueue kernels and return; nothing synchronises.
 *   - A non-ATTN_OK return from argument validation means nothing was
 *     enqueued and no output was touched.
 *   - LSE is the natural-log log-sum-exp of the scaled scores of the row's
 *     valid keys: lse = m + ln(l).  A row with no valid key has O = 0 and
 *     lse = -inf.
 *   - Causal masking is the lower-triangular mask aligned to the bottom
 *     right: key j is visible to query i iff j <= i + (Nk - Nq) (the pages'
 *     "下三角" mask, Capstone page section 7.3; identical to j <= i when
 *     Nq == Nk).
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* NULL pointer, non-positive size, misalignment, bad scale */
    ATTN_ERR_UNSUPPORTED = 2,  /* a head dim / page size / dtype this build has no kernel for */
    ATTN_ERR_CUDA = 3,         /* a CUDA runtime call or a kernel launch failed */
    ATTN_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than the size query asked for */
    ATTN_ERR_TIMEOUT = 5,      /* a kernel's bounded wait gave up (device status word) */
    ATTN_ERR_DEVICE_DATA = 6   /* a device-side length or page id was out of range (status word) */
} attn_status_t;

/* Dense prefill, bf16.
 *   q: bf16 [B, H, Nq, d]; k, v: bf16 [B, H, Nk, d]   (read only)
 *   o: bf16 [B, H, Nq, d]                               (written)
 *   lse: fp32 [B, H, Nq] or NULL                        (written when non-NULL)
 *   d in {64, 128}; B, H, Nq, Nk >= 1; B*H < 2^31; scale finite and > 0
 *   (1/sqrt(d) for standard attention); causal 0 or 1.
 * Output rounding: O is rounded once from fp32 to bf16 (nearest-even).
 * Errors: ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED before any launch;
 * ATTN_ERR_CUDA when the launch fails. */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int Nq, int Nk, int d, float scale, int causal,
                       void* stream);

/* Dense prefill on FP8-e4m3fn inputs ("Flash Attention 3 指南", the FP8
 * path: e4m3 operands, fp32-accumulated products, P cast to e4m3 before the
 * P*V product, 16-bit output).
 *   q8, k8, v8: e4m3fn codes, [B, H, Nq|Nk, d] like attn_fwd;
 *   q_descale, k_descale, v_descale: per-tensor factors, the real value of a
 *   code x is decode(x) * descale (with per-tensor amax scaling the descale
 *   is amax / 448);
 *   o: bf16 [B, H, Nq, d]; lse: fp32 [B, H, Nq] or NULL.
 *   Scores are scale * q_descale * k_descale * (q8 . k8); the unnormalised
 *   probabilities are rounded to e4m3 (nearest, saturating) before the P*V
 *   product while l sums them in fp32; O = v_descale * (P8 V8) / l.
 *   d must be 128.  Errors as attn_fwd. */
attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v8,
                           float q_descale, float k_descale, float v_descale,
                           void* o, float* lse,
                           int B, int H, int Nq, int Nk, int d, float scale, int causal,
                           void* stream);

/* Bytes of device workspace attn_paged_decode needs for these sizes
 * (0 on invalid sizes).  The workspace holds the per-split partial results
 * (unnormalised O, m, l) that the merge step combines.
 * NOTE the argument order: max_pages_per_seq comes BEFORE page_size here,
 * the reverse of attn_paged_decode's own (..., page_size, max_pages_per_seq,
 * ...).  Both are int, so swapping them is not caught by the compiler. */
size_t attn_paged_decode_workspace_size(int B, int H, int d, int max_pages_per_seq, int page_size);

/* One-token decode over a paged KV cache ("FlashAttention V3 实战", section
 * 3.2: vLLM/SGLang-style page tables).  Each request's keys are split into
 * chunks of pages that are processed independently; the partial results are
 * combined with the (m, l, O) merge of the Capstone page, section 2.2 step 4:
 *   m = max_s m_s,  l = sum_s l_s e^(m_s - m),  O = sum_s e^(m_s - m) O_s / l.
 *   q: bf16 [B, H, d] (one query token per request)
 *   k_cache, v_cache: bf16 [num_pages, page_size, H, d]
 *   block_table: int32 [B, max_pages_per_seq], physical page ids
 *   seq_lens: int32 [B], keys 0..seq_lens[r]-1 of request r are attended;
 *     key t lives at cache[block_table[r][t / page_size]][t % page_size]
 *   o: bf16 [B, H, d]; lse: fp32 [B, H] or NULL
 *   workspace: device buffer of at least
 *     attn_paged_decode_workspace_size(B, H, d, max_pages_per_seq, page_size)
 *     bytes, owned by the caller, contents need no initialisation.
 *   d in {64, 128}; page_size a multiple of 8 in [8, 1024].
 * Device-side data (seq_lens, block_table) is the caller's contract: a
 * length outside [0, max_pages_per_seq*page_size] is clamped and a page id
 * outside [0, num_pages) is skipped; either sets the device status word to
 * ATTN_ERR_DEVICE_DATA (read it with attn_device_status). */
attn_status_t attn_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens,
                                int B, int H, int d, int page_size, int max_pages_per_seq,
                                int num_pages, float scale, void* o, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Size of the fixed device scratch array used by attn_paged_decode_noalloc. */
#define ATTN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* Paged decode without any allocation (no counterpart on the attention pages:
 * an addition for callers).  Some callers cannot allocate device memory at
 * call time: a serving loop whose device memory is fully reserved up front
 * for its own KV-cache pool, or one that forbids cudaMalloc after start-up
 * because it can synchronise the device and stall other streams.  This entry
 * point takes the same arguments as attn_paged_decode minus the workspace and
 * computes the same result; the split partials live in a fixed device array
 * of ATTN_NOALLOC_SCRATCH_BYTES owned by the library, which every GPU that
 * loads the library holds until the process exits.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (on
 *     different streams, or from different host threads without ordering)
 *     race and give undefined results.  Partials from an earlier call are
 *     never read, so nothing needs clearing between calls.
 *   - If the partials do not fit, the split is coarsened (more pages per
 *     split); if even one split per request exceeds the array, the call
 *     returns ATTN_ERR_WORKSPACE and enqueues nothing.
 *   - Nothing is allocated or freed: no cudaMalloc, cudaFree or allocating
 *     library routine is called.
 * Other errors and the device-data contract are as for attn_paged_decode. */
attn_status_t attn_paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        int B, int H, int d, int page_size, int max_pages_per_seq,
                                        int num_pages, float scale, void* o, float* lse, void* stream);

/* Bytes of device workspace attn_paged_fwd needs for these sizes (0 on
 * invalid sizes): a work list (which work units have keys to process, built
 * by each call on `stream`, and the counter its CTAs take entries with) and,
 * when a request's keys are split over several CTAs, the per-split partials
 * (unnormalised O, m, l). */
size_t attn_paged_fwd_workspace_size(int B, int total_q, int max_q_len, int H, int H_kv, int d, int page_size,
                                     int max_pages_per_seq);

/* Attention over a paged KV cache on the tensor cores, for grouped-query
 * decode and for prefill chunks appended to cached prefixes.
 * The cache is the page-table layout of "FlashAttention V3 实战", section 3.2,
 * with H_kv KV heads per slot; query head h reads KV head h / (H / H_kv)
 * (grouped-query attention; H_kv = H is multi-head, H_kv = 1 multi-query).
 * The arithmetic is that of attn_fwd: online softmax (Capstone page, section
 * 2.2) with one final division, and the (m, l, O) merge of section 2.2 step 4
 * when a request's keys are split over several CTAs.
 *   q: bf16 [total_q, H, d], token-major: request r owns query tokens
 *     cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1
 *   k_cache, v_cache: bf16 [num_pages, page_size, H_kv, d]
 *   block_table: int32 [B, max_pages_per_seq], physical page ids
 *   cu_seqlens_q: int32 [B + 1] device offsets, non-decreasing, first 0 and
 *     last total_q, each request at most max_q_len tokens; or NULL for one
 *     query token per request (then total_q == B and max_q_len == 1)
 *   seq_lens: int32 [B] device key counts; the request's query tokens are its
 *     last q_len keys (their K/V already written to the cache), so query i of
 *     request r sits at position seq_lens[r] - q_len_r + i; key t lives at
 *     cache[block_table[r][t / page_size]][t % page_size]
 *   causal: 1 = query at position P sees keys t <= P (the bottom-right
 *     aligned lower triangle of attn_fwd); 0 = every query sees all keys
 *   o: bf16 [total_q, H, d]; lse: fp32 [total_q, H] or NULL
 *   workspace: at least attn_paged_fwd_workspace_size(...) bytes,
 *     caller-owned, 16-byte aligned, contents need no initialisation; calls
 *     that may overlap on the GPU need distinct workspaces
 *   d in {64, 128}; page_size a power of two in [8, 1024]; H % H_kv == 0 and
 *   H / H_kv <= 128.
 * A query with no visible key gets O = 0 and lse = -inf.
 * Device-side data is the caller's contract: offsets out of range drop that
 * request's queries (its rows are not written), a length outside
 * [0, max_pages_per_seq * page_size] is clamped, a page id outside
 * [0, num_pages) reads zeros; each sets the device status word to
 * ATTN_ERR_DEVICE_DATA, after which the call's results are undefined.
 * Errors: ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED / ATTN_ERR_WORKSPACE
 * before any launch; ATTN_ERR_CUDA when a launch fails. */
attn_status_t attn_paged_fwd(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                             int B, int total_q, int max_q_len, int H, int H_kv, int d, int page_size,
                             int max_pages_per_seq, int num_pages, float scale, int causal,
                             void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace attn_varlen_fwd needs (0 on invalid sizes); the
 * same layout as for attn_paged_fwd. */
size_t attn_varlen_fwd_workspace_size(int B, int total_q, int max_q_len, int max_k_len, int H, int H_kv, int d);

/* Variable-length batch prefill: B independent attention problems packed
 * back to back without padding, grouped KV heads as in attn_paged_fwd (the
 * same kernel, reading K/V rows directly instead of through a page table).
 *   q: bf16 [total_q, H, d]; request r owns query rows
 *     cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1
 *   k, v: bf16 [total_k, H_kv, d]; request r owns key rows
 *     cu_seqlens_k[r] .. cu_seqlens_k[r+1]-1
 *   cu_seqlens_q, cu_seqlens_k: int32 [B + 1] device offsets, non-decreasing,
 *     first 0 and last total_q / total_k; per request at most max_q_len
 *     queries and max_k_len keys
 *   causal: 1 = query i of a request with q_len queries and k_len keys sees
 *     keys t <= i + (k_len - q_len) (the bottom-right aligned lower triangle
 *     of attn_fwd); 0 = every query sees all of its request's keys
 *   o: bf16 [total_q, H, d]; lse: fp32 [total_q, H] or NULL
 *   workspace: at least attn_varlen_fwd_workspace_size(...) bytes,
 *     caller-owned, 16-byte aligned, no initialisation needed
 *   d in {64, 128}; H % H_kv == 0 and H / H_kv <= 128.
 * A query with no visible key gets O = 0 and lse = -inf.  Offsets out of
 * range set the device status word to ATTN_ERR_DEVICE_DATA (the call's
 * results are then undefined).  Errors as attn_paged_fwd. */
attn_status_t attn_varlen_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, int B, int total_q, int total_k, int max_q_len,
                              int max_k_len, int H, int H_kv, int d, float scale, int causal, void* o,
                              float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace attn_bwd needs (0 on invalid sizes): an fp32 dQ
 * accumulator and two fp32 row vectors, padded to whole 128-row blocks. */
size_t attn_bwd_workspace_size(int B, int H, int Nq, int d);

/* Backward pass of attn_fwd: dQ, dK, dV of O = softmax(scale Q K^T) V for
 * the upstream gradient dO, recomputing the probabilities from Q, K and the
 * forward pass's LSE instead of storing them ("Capstone" page, section 6.1,
 * the pitfalls table: keep m, l and recompute; section 7.3, question 1):
 *   P = exp(scale Q K^T - lse),  D = rowsum(dO * O),  dS = P * (dO V^T - D),
 *   dV = P^T dO,  dQ = scale dS K,  dK = scale dS^T Q.
 *   q, o, dout: bf16 [B, H, Nq, d]; k, v: bf16 [B, H, Nk, d]; lse: fp32
 *   [B, H, Nq], all as produced / consumed by attn_fwd with the same scale
 *   and causal flag (read only); dq: bf16 [B, H, Nq, d], dk, dv: bf16
 *   [B, H, Nk, d] (written).  P and dS enter the tensor-core products as
 *   bf16, accumulation is fp32, dQ is accumulated across key blocks in fp32
 *   and rounded once.  Rows with lse = -inf (no visible key) get dQ = 0;
 *   keys no query sees get dK = dV = 0.
 *   workspace: attn_bwd_workspace_size(B, H, Nq, d) bytes, caller-owned,
 *   16-byte aligned, no initialisation needed.
 *   d in {64, 128}; B * H <= 65535 and B * H * ceil(Nk / 128) < 2^31
 *   (else ATTN_ERR_UNSUPPORTED).  Errors as attn_fwd, plus
 *   ATTN_ERR_WORKSPACE. */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                       float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace attn_fwd_host needs (0 on invalid sizes): three
 * chunk slots, each holding one chunk of Q, K, V and, per mask mode, one
 * chunk of O and LSE.  chunk_bh <= 0 asks for the default chunk. */
size_t attn_fwd_host_workspace_size(int B, int H, int Nq, int Nk, int d, int n_modes, int chunk_bh);

/* Dense bf16 prefill with the inputs and outputs in HOST memory: the
 * attn_fwd computation for each of n_modes mask modes over the same Q, K, V,
 * with the host<->device copies inside the call.
 *   q: host bf16 [B, H, Nq, d]; k, v: host bf16 [B, H, Nk, d]   (read only)
 *   causal[i] in {0, 1} for i < n_modes, 1 <= n_modes <= 8;
 *   o[i]: host bf16 [B, H, Nq, d]; lse[i]: host fp32 [B, H, Nq] or NULL.
 *   chunk_bh: batch-head pairs per chunk (<= 0: about an eighth of B*H).
 *   workspace: DEVICE memory of attn_fwd_host_workspace_size() bytes,
 *   16-byte aligned.
 * The (b, h) range is cut into chunks of chunk_bh pairs.  Each chunk is
 * copied in on one internal stream, computed on `stream` (one attn_fwd
 * kernel per mode), and copied out on a second internal stream, so the two
 * copy directions and the kernels of neighbouring chunks overlap.  Each
 * (b, h) problem is computed by the same kernel as attn_fwd, so the outputs
 * are bit-identical to attn_fwd on device copies of the inputs.  The copies
 * overlap only when the host buffers are page-locked (cudaHostAlloc or
 * cudaHostRegister); pageable buffers give the same results serially.
 * Ordering: the copies start after the work already enqueued on `stream`;
 * work enqueued on `stream` after the call starts after every output has
 * landed in host memory.  Synchronise `stream` before reading the outputs.
 * Resources: the first call on a device creates two streams and ten events
 * there, kept for the life of the process.  Calls on one device are
 * serialised by a host lock while they enqueue.
 * Errors: ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED / ATTN_ERR_WORKSPACE
 * before anything is enqueued (also when a pointer is device memory);
 * ATTN_ERR_CUDA if a copy or launch fails part-way (outputs undefined). */
attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, int n_modes, const int* causal,
                            void* const* o, float* const* lse, int B, int H, int Nq, int Nk, int d, float scale,
                            int chunk_bh, void* workspace, size_t workspace_bytes, void* stream);

/* Failure-handling check: launches a one-warp kernel whose bounded wait --
 * the same wait every attention kernel uses -- is on a barrier that nothing
 * completes.  After the wait limit (2 s) it gives up and records
 * ATTN_ERR_TIMEOUT in the device status word, as a stalled attention kernel
 * would; nothing faults or hangs and the context stays usable.  While the
 * timeout is recorded the attention kernels return without work (see
 * attn_device_status).  Errors: ATTN_ERR_CUDA if the launch fails. */
attn_status_t attn_selftest_wait_timeout(void* stream);

/* Dense tensor-core rate check (no counterpart on the attention pages: the
 * denominator of the prefill roofline, measured rather than quoted).
 * Launches n_ctas CTAs of 128 threads, each large enough in shared memory to
 * have an SM to itself (launch one per SM).  One thread per CTA issues
 * 4 * n_groups back-to-back tcgen05.mma of M = N = 128, K = 16, bf16
 * operands from shared memory, fp32 accumulation into tensor memory (the
 * pattern of S = Q K^T), and writes the SM cycles they took (clock64, from
 * the first issue to completion) to cycles[cta].  Each MMA is
 * 2 * 128 * 128 * 16 FLOP, so FLOP per SM cycle = 524288 * n_groups /
 * cycles[cta]; x SM count x SM clock = the device's dense bf16 rate.
 *   cycles: DEVICE array of n_ctas uint64, 8-byte aligned (written; 0 for a
 *   CTA whose bounded wait gave up, which also sets ATTN_ERR_TIMEOUT).
 *   1 <= n_ctas <= 65535, 1 <= n_groups <= 2^20.
 * Errors: ATTN_ERR_INVALID_ARG before the launch; ATTN_ERR_CUDA if it fails. */
attn_status_t attn_selftest_mma_rate(unsigned long long* cycles, int n_ctas, int n_groups, void* stream);

/* Synchronises `stream`, then reads and clears the calling device's status
 * word in one atomic step (a one-thread kernel on `stream`; a bit another
 * stream's kernel sets meanwhile is kept for the next call, never lost).
 * Kernels set the word when a bounded internal wait gives up
 * (ATTN_ERR_TIMEOUT; the kernel then returns early and its outputs are
 * undefined) or when device-side lengths, offsets or page ids are out of
 * range (ATTN_ERR_DEVICE_DATA; the kernel clamps them, carries on, and the
 * call's results are undefined).
 * While a TIMEOUT is recorded, every attention kernel of the device returns
 * without work -- those launched later, and those already running on any
 * stream, at their next internal wait -- so a stalled device goes quiet.
 * DEVICE_DATA cancels nothing: it only reports the call that found the bad
 * data.  Check the word after any call whose result matters.
 * Returns ATTN_OK, one of those two codes (TIMEOUT first when both are set),
 * or ATTN_ERR_CUDA. */
attn_status_t attn_device_status(void* stream);

/* Static English description of a status code (never NULL). */
const char* attn_status_string(attn_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
