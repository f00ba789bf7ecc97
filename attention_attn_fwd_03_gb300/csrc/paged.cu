// paged.cu -- exact attention over a paged KV cache on the tensor cores:
// grouped-query decode and prefill chunks appended to cached prefixes; the
// same kernel also takes contiguous ragged K/V (variable-length batch
// prefill, key t of request r at row cu_k[r] + t).
//
// The cache is the block-table layout of "FlashAttention V3 实战: Hopper 架构下
// 的 Paged KV Cache 协同优化", section 3.2 (fixed-size pages named by a
// per-request table, the vLLM / SGLang layout), here with H_kv KV heads per
// slot; query head h reads KV head h / G, G = H / H_kv.  The arithmetic is the
// one-pass online softmax of "Capstone: CUDA Softmax 与 Attention 算子",
// sections 2.2 and 4.1-4.2 (running max m, denominator l, unnormalised O
// rescaled by 2^(m_old - m_new), one final division), in log2 units.
//
// Packing: the G query heads that share a KV head are the rows of one query
// tile, together with up to T = 128 / G consecutive query tokens of the same
// request (row = t * G + g).  Grouped decode thus becomes a [G x d] x [d x 128]
// product per key block that the 128-row tensor-core MMA takes whole, and the
// K/V bytes of a KV head are read once for all G heads.  A prefill chunk
// fills the tile with T tokens.
//
// Work unit = (request, KV head, query tile, split); a split is a run of
// split_blocks KV blocks of 128 keys.  With more than one split the units
// write unnormalised partials (O_s, m_s, l_s) and a merge kernel combines
// them with the (m, l, O) merge of the Capstone page, section 2.2 step 4.
// Request lengths live on the device, so a one-CTA schedule pass first lists
// the units that have work, longest first; the persistent CTAs then take
// list entries from an atomic counter (work units differ in size by up to the split length, and
// dynamic fetching keeps the SMs evenly loaded to the end).
//
// Persistent CTAs (one per SM), 192 threads:
//   warp 0    TMA producer: per unit the Q tile (box: 64 dims x G heads x T
//             tokens), then K_j, V_j of every KV block into an NST-stage ring.
//             A block of 128 keys is gathered from 128 / R page boxes of R
//             rows (R = min(page_size, 128)); the warp's lanes fetch 32 page
//             ids at a time from the block table.  Boxes past the request's
//             keys, or naming an out-of-range page, read the zero fill past
//             the end of the cache.
//   warp 1    MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM S
//             buffers, O += P_j V_j with P_j read from TMEM.  S_{j+1} is issued
//             before PV_j so the next block's scores are computed while the
//             softmax works on the current one.
//   warps 2-5 softmax: one thread per tile row; masks (request length, causal
//             position), updates (m, l) with lazy rescaling (threshold kTau),
//             writes P as bf16 over S, rescales O after PV_{j-1} completed, and
//             zeroes the V rows of a partial last page (cache slots past the
//             request's length may hold anything, and 0 * NaN would poison
//             the P V product); then the epilogue writes O / l (or the
//             partials) and the LSE row by row.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace attn {

namespace {

constexpr float kTau = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

constexpr int kQN = 4;        // unit-queue slots between the producer and the other roles
constexpr int kSlotInts = 11;  // one decoded unit per slot (see publish_unit)

template <int D>
struct PCfg {
    static constexpr int NPANEL = D / 64;          // 128-byte panels of the head dim
    static constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B
    static constexpr int TILE_BYTES = NPANEL * PANEL_BYTES;
    static constexpr int NST = D == 128 ? 5 : 8;   // K/V ring stages
    static constexpr uint32_t TM_O = 256;          // S buffers at columns 0 and 128
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int OFF_Q = 0;                // two Q tiles
    static constexpr int OFF_KV = OFF_Q + 2 * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_KV + NST * TILE_BYTES;
    static constexpr int N_BARS = 2 * NST + 11 + 2 * kQN;
    static constexpr int OFF_UQ = OFF_BAR + 8 * N_BARS;
    static constexpr int OFF_MISC = OFF_UQ + 4 * kQN * kSlotInts;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // more than half an SM's shared memory: one CTA per SM owns all 512 TMEM columns
    static constexpr int SMEM_BYTES = (SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024);
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct PBars {
    uint64_t* q_full;    // [2], one per Q buffer
    uint64_t* q_empty;   // [2]
    uint64_t* kv_full;   // [NST]
    uint64_t* kv_empty;  // [NST]
    uint64_t* s_full;    // [2], one per S buffer
    uint64_t* p_full;    // 128 arrivals per block
    uint64_t* o_full;    // one phase per PV product
    uint64_t* o_empty;   // 128 arrivals per unit
    uint64_t* done;
    uint64_t* uq_full;   // [kQN], the producer published a unit into the slot
    uint64_t* uq_empty;  // [kQN], 5 arrivals: the MMA issuer and the four softmax warps read it
};

struct PUnit {
    int r, kvh, split;
    int q_start, q_len, kv_len;
    int t0, nt;   // the tile's tokens [t0, t0 + nt) of the request; nt <= 0: no tile
    int kb0, nb;  // the unit's KV blocks [kb0, kb0 + nb)
    bool bad;     // the request's offsets or length were out of range
};

// Query tokens and key count of request r, checked against the launch's
// bounds.  Offsets out of range drop the request's queries (q_len = 0); a
// length out of range is clamped.  Either marks the unit bad.
__device__ __forceinline__ void request_extent(const PagedParams& p, int r, PUnit& g) {
    g.bad = false;
    if (p.cu_q != nullptr) {
        const int a = __ldg(p.cu_q + r), b = __ldg(p.cu_q + r + 1);
        g.q_start = a;
        g.q_len = b - a;
        if (a < 0 || b < a || b > p.total_q || g.q_len > p.max_q_len) {
            g.bad = true;
            g.q_start = 0;
            g.q_len = 0;
        }
    } else {
        g.q_start = r;
        g.q_len = 1;
    }
    const int cap = p.max_pages * p.page_size;
    if (p.cu_k != nullptr) {  // contiguous keys: rows cu_k[r] .. cu_k[r+1] - 1
        const int a = __ldg(p.cu_k + r), b = __ldg(p.cu_k + r + 1);
        g.kv_len = b - a;
        if (a < 0 || b < a || b > p.kv_rows) {
            g.bad = true;
            g.kv_len = 0;
        }
    } else {
        g.kv_len = __ldg(p.seq_lens + r);
    }
    if (g.kv_len < 0 || g.kv_len > cap) {
        g.bad = true;
        g.kv_len = g.kv_len < 0 ? 0 : cap;
    }
}

// KV blocks visible to a tile of a request whose last token is t_last: all
// keys, or under the causal mask the keys up to that token's position
// kv_len - q_len + t_last (bottom-right alignment).
__device__ __forceinline__ int tile_kv_blocks(const PagedParams& p, int q_len, int kv_len, int t_last) {
    long long key_end = kv_len;
    if (p.causal) {
        key_end = (long long)kv_len - q_len + t_last + 1;
        if (key_end > kv_len) key_end = kv_len;
    }
    if (key_end <= 0) return 0;
    return (int)((key_end + 127) / 128);
}

// Unit u: KV head fastest, then request, then query tile (last tiles, the
// heaviest under the causal mask, first), then split.  unit_tile fills in
// the tile and its KV blocks once the request's extent is in g.
__device__ __forceinline__ void unit_tile(const PagedParams& p, int u, PUnit& g) {
    g.kvh = u % p.H_kv;
    int x = u / p.H_kv;
    g.r = x % p.B;
    x /= p.B;
    const int qt = p.n_qt - 1 - x % p.n_qt;
    g.split = x / p.n_qt;
    g.t0 = qt * p.T;
    g.nt = min(p.T, g.q_len - g.t0);
    const int nb_all = g.nt > 0 ? tile_kv_blocks(p, g.q_len, g.kv_len, g.t0 + g.nt - 1) : 0;
    g.kb0 = g.split * p.split_blocks;
    g.nb = max(0, min(p.split_blocks, nb_all - g.kb0));
}

// A listed unit id with this bit set covers all of its request's KV blocks
// (the request is not split: its unit writes O and the LSE itself).
constexpr int kWholeBit = 1 << 30;

// A whole request's unit: every KV block of its tile, no split.
__device__ __forceinline__ void make_whole(const PagedParams& p, PUnit& g) {
    g.split = -1;
    g.kb0 = 0;
    g.nb = g.nt > 0 ? tile_kv_blocks(p, g.q_len, g.kv_len, g.t0 + g.nt - 1) : 0;
}

__device__ __forceinline__ PUnit paged_unit(const PagedParams& p, int u) {
    PUnit g;
    request_extent(p, (u / p.H_kv) % p.B, g);
    unit_tile(p, u, g);
    return g;
}

// Queue slots carry the unit already decoded, so that the MMA issuer and the
// softmax warps start a unit without global loads on their critical path.
__device__ __forceinline__ void publish_unit(volatile int* q, int u, const PUnit& g) {
    q[0] = u;
    q[1] = g.r;
    q[2] = g.kvh;
    q[3] = g.split;
    q[4] = g.q_start;
    q[5] = g.q_len;
    q[6] = g.kv_len;
    q[7] = g.t0;
    q[8] = g.nt;
    q[9] = g.kb0;
    q[10] = g.nb;
}

__device__ __forceinline__ int read_unit(const volatile int* q, PUnit& g) {
    g.r = q[1];
    g.kvh = q[2];
    g.split = q[3];
    g.q_start = q[4];
    g.q_len = q[5];
    g.kv_len = q[6];
    g.t0 = q[7];
    g.nt = q[8];
    g.kb0 = q[9];
    g.nb = q[10];
    g.bad = false;
    return q[0];
}

__device__ __forceinline__ void st_global_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// ---------------------------------------------------------------- producer (whole warp)

template <int D>
__device__ void producer_role(const PagedParams& p, uint8_t* smem, const PBars& b, volatile int* uq,
                              volatile int* abort_flag, int lane) {
    using C = PCfg<D>;
    if (lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
    }
    const int R = p.rows_per_box;
    const int LPB = 128 / R;                    // boxes per panel per KV block (1..16)
    const int oob = p.kv_rows;  // first row past the K/V tensor: zero fill
    int kv_idx = 0, qcnt = 0, pub = 0;
    bool ok = true;
    // the schedule pass listed the units with work; take them in list order
    // The list built by the schedule pass (entries: unit, q_start, q_len,
    // kv_len) is taken in order: entry blockIdx.x first (read alongside the
    // list length; the entry exists since the grid is no larger than the unit
    // count), then entries gridDim.x, gridDim.x + 1, ... through the fetch
    // counter.  The next entry is fetched while the current unit's loads are
    // issued, and no further global load is needed to decode it.
    griddep_wait();  // the list exists once the schedule pass has completed
    const int total = p.sched[1];
    int4 next = make_int4(-1, 0, 0, 0);
    if (lane == 0) {
        const int4 e = p.sched_list[blockIdx.x];
        if ((int)blockIdx.x < total) next = e;
    }
    for (;;) {
        int4 cur;
        cur.x = __shfl_sync(0xffffffffu, next.x, 0);
        cur.y = __shfl_sync(0xffffffffu, next.y, 0);
        cur.z = __shfl_sync(0xffffffffu, next.z, 0);
        cur.w = __shfl_sync(0xffffffffu, next.w, 0);
        const int u = cur.x < 0 ? -1 : (cur.x & ~kWholeBit);
        const bool more = u >= 0;
        if (more && lane == 0) {
            const int k = (int)gridDim.x + atomicAdd(p.sched, 1);
            next = k < total ? p.sched_list[k] : make_int4(-1, 0, 0, 0);
        }
        PUnit g{};
        if (more) {
            g.q_start = cur.y;
            g.q_len = cur.z;
            g.kv_len = cur.w;
            g.bad = false;
            unit_tile(p, u, g);
            if (cur.x & kWholeBit) make_whole(p, g);
        }
        // publish the unit (or the end mark) to the MMA issuer and the softmax warps
        if (lane == 0) {
            const int slot = pub % kQN;
            if (pub >= kQN) ok = wait_bar(&b.uq_empty[slot], (uint32_t)((pub / kQN - 1) & 1), abort_flag, p.status);
            if (ok) {
                publish_unit(uq + slot * kSlotInts, more ? u : -1, g);
                bar_arrive(&b.uq_full[slot]);  // release: the slot's value is visible to the waiters
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok || !more) break;
        ++pub;
        if (g.nb == 0) continue;  // only the softmax warps act (zero rows)
        // the query tile into buffer qcnt & 1, released by the unit two back
        const int qb = qcnt & 1;
        if (lane == 0) {
            if (qcnt >= 2) ok = wait_bar(&b.q_empty[qb], (uint32_t)(((qcnt >> 1) - 1) & 1), abort_flag, p.status);
            if (ok) {
                bar_arrive_expect_tx(&b.q_full[qb], p.q_tile_bytes);
#pragma unroll
                for (int pn = 0; pn < C::NPANEL; ++pn)
                    tma_load_3d(smem + C::OFF_Q + qb * C::TILE_BYTES + pn * C::PANEL_BYTES, &p.tm_q, &b.q_full[qb],
                                pn * 64, g.kvh * p.G, g.q_start + g.t0);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++qcnt;  // counts issued loads only: the drain below waits for each
        // K and V blocks; lane i holds the cache row of box (batch * 32 + i):
        // through the block table, or cu_k[r] + key for contiguous keys
        const long long key0 = (long long)g.kb0 * 128;
        const int n_boxes = g.nb * LPB;
        const int kst = p.cu_k != nullptr ? min(max(__ldg(p.cu_k + g.r), 0), oob) : 0;
        int my_row = oob;
        for (int j = 0; ok && j < g.nb; ++j) {
            const int box0 = j * LPB;
            if ((box0 & 31) == 0) {
                const int bi = box0 + lane;
                int row = oob;
                if (bi < n_boxes) {
                    const long long key = key0 + (long long)bi * R;
                    if (key < g.kv_len) {
                        if (p.cu_k != nullptr) {
                            row = kst + (int)key;
                        } else {
                            const int pg = (int)(key / p.page_size);
                            const int id = __ldg(p.block_table + (size_t)g.r * p.max_pages + pg);
                            if (id >= 0 && id < p.num_pages)
                                row = id * p.page_size + (int)(key % p.page_size);
                            else
                                atomicOr(p.status, 1u << kStatusDeviceData);
                        }
                    }
                }
                my_row = row;
            }
            int rows[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) rows[i] = __shfl_sync(0xffffffffu, my_row, (box0 + (i < LPB ? i : 0)) & 31);
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                if (lane == 0) {
                    const int slot = kv_idx % C::NST, round = kv_idx / C::NST;
                    if (round > 0) ok = wait_bar(&b.kv_empty[slot], (uint32_t)((round - 1) & 1), abort_flag, p.status);
                    if (ok) {
                        bar_arrive_expect_tx(&b.kv_full[slot], C::TILE_BYTES);
                        const CUtensorMap* map = kv ? &p.tm_v : &p.tm_k;
                        uint8_t* dst = smem + C::OFF_KV + slot * C::TILE_BYTES;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (i >= LPB) break;
#pragma unroll
                            for (int pn = 0; pn < C::NPANEL; ++pn)
                                tma_load_3d(dst + pn * C::PANEL_BYTES + i * R * 128, map, &b.kv_full[slot], pn * 64,
                                            g.kvh, rows[i]);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                ++kv_idx;
            }
        }
        if (!ok) break;
    }
    // Drain: every copy this warp started must land before the CTA exits.
    if (lane == 0) {
        for (int i = qcnt - 2 > 0 ? qcnt - 2 : 0; i < qcnt; ++i)
            drain_wait(&b.q_full[i & 1], (uint32_t)((i >> 1) & 1), p.status);
        for (int idx = kv_idx - C::NST > 0 ? kv_idx - C::NST : 0; idx < kv_idx; ++idx)
            drain_wait(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), p.status);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- MMA issuer (one thread)

template <int D>
__device__ void mma_role(const PagedParams& p, uint8_t* smem, const PBars& b, volatile int* uq,
                         volatile int* abort_flag, uint32_t tmem) {
    using C = PCfg<D>;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t kv0 = sbase + C::OFF_KV;
    auto k_desc = [&](int idx) { return sdesc_sw128(kv0 + (uint32_t)((idx % C::NST) * C::TILE_BYTES), 16, 1024); };
    auto v_desc = [&](int idx) {
        return sdesc_sw128(kv0 + (uint32_t)((idx % C::NST) * C::TILE_BYTES), C::PANEL_BYTES, 1024);
    };
    auto wait_full = [&](int idx) {
        return wait_bar(&b.kv_full[idx % C::NST], (uint32_t)((idx / C::NST) & 1), abort_flag, p.status);
    };
    const uint32_t d_o = tmem + C::TM_O;
    int kv_base = 0, qcnt = 0, units = 0;
    uint32_t sblk = 0;  // KV blocks processed so far: block sblk uses S buffer sblk & 1
    for (int k = 0;; ++k) {
        const int slot = k % kQN;
        if (!wait_bar(&b.uq_full[slot], (uint32_t)((k / kQN) & 1), abort_flag, p.status)) return;
        PUnit g;
        const int u = read_unit(uq + slot * kSlotInts, g);
        bar_arrive(&b.uq_empty[slot]);
        if (u < 0) break;
        const int nb = g.nb;
        if (nb == 0) continue;
        const int qb = qcnt & 1;
        if (!wait_bar(&b.q_full[qb], (uint32_t)((qcnt >> 1) & 1), abort_flag, p.status)) return;
        ++qcnt;
        const uint64_t q_desc = sdesc_sw128(sbase + (uint32_t)(C::OFF_Q + qb * C::TILE_BYTES), 16, 1024);
        if (!wait_full(kv_base)) return;
        tc_fence_after();
        issue_s<D, false>(tmem + (sblk & 1u) * 128u, q_desc, k_desc(kv_base));
        tc_commit(&b.s_full[sblk & 1u]);
        tc_commit(&b.kv_empty[kv_base % C::NST]);
        if (nb == 1) tc_commit(&b.q_empty[qb]);
        for (int j = 0; j < nb; ++j) {
            const uint32_t sb = sblk + (uint32_t)j;
            const int iV = kv_base + 2 * j + 1, iK1 = kv_base + 2 * j + 2;
            if (j + 1 < nb) {  // S_{j+1} into the other buffer (its P_{j-1} was consumed by PV_{j-1})
                if (!wait_full(iK1)) return;
                tc_fence_after();
                issue_s<D, false>(tmem + ((sb + 1u) & 1u) * 128u, q_desc, k_desc(iK1));
                tc_commit(&b.s_full[(sb + 1u) & 1u]);
                tc_commit(&b.kv_empty[iK1 % C::NST]);
                if (j + 1 == nb - 1) tc_commit(&b.q_empty[qb]);
            }
            if (!wait_full(iV)) return;
            if (j == 0 && units > 0 && !wait_bar(b.o_empty, (uint32_t)((units - 1) & 1), abort_flag, p.status))
                return;
            if (!wait_bar(b.p_full, sb & 1u, abort_flag, p.status)) return;
            tc_fence_after();
            issue_pv<D, false>(d_o, tmem + (sb & 1u) * 128u, v_desc(iV), j > 0);
            tc_commit(b.o_full);
            tc_commit(&b.kv_empty[iV % C::NST]);
        }
        sblk += (uint32_t)nb;
        kv_base += 2 * nb;
        ++units;
    }
}

// ---------------------------------------------------------------- softmax + epilogue

template <int D>
__device__ void softmax_role(const PagedParams& p, uint8_t* smem, const PBars& b, volatile int* uq,
                             volatile int* abort_flag, uint32_t tmem, int wq, int lane) {
    using C = PCfg<D>;
    const int row = wq * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::TM_O;
    const float cs = p.c_scale;
    const int tr = row / p.G, gh = row % p.G;  // token within the tile, head within the group
    const uint32_t kv_smem = smem_u32(smem + C::OFF_KV);
    uint32_t sblk = 0, ocnt = 0;
    int kv_base = 0;
    bool ok = true;

    for (int k = 0; ok; ++k) {
        const int slot = k % kQN;
        ok = __all_sync(0xffffffffu, wait_bar(&b.uq_full[slot], (uint32_t)((k / kQN) & 1), abort_flag, p.status));
        if (!ok) break;
        PUnit g;
        const int u = read_unit(uq + slot * kSlotInts, g);
        __syncwarp();
        if (lane == 0) bar_arrive(&b.uq_empty[slot]);
        if (u < 0) break;
        if (g.nt <= 0) continue;
        const bool row_ok = tr < g.nt;
        // Every row of this warp is padding (a decode tile fills G of its 128 rows): its scores are
        // not needed, so it skips their exponentials; the PV product then reads stale values in
        // those rows, which touch only those rows of O, never stored.
        const bool idle = wq * 32 >= g.nt * p.G;
        const int head = g.kvh * p.G + gh;
        const size_t grow = (size_t)(g.q_start + g.t0 + (row_ok ? tr : 0)) * p.H + head;  // output row
        if (g.nb == 0) {  // no visible key: O = 0, LSE = -inf (split partials: the merge sees no split)
            if ((p.n_splits == 1 || g.split < 0) && row_ok) {
                uint16_t* dst = p.o + grow * D;
#pragma unroll
                for (int c = 0; c < D; c += 8) st_global_v4(dst + c, 0u, 0u, 0u, 0u);
                if (p.lse != nullptr) p.lse[grow] = -INFINITY;
            }
            continue;
        }
        const long long kv_len = g.kv_len;
        const long long pos0 = kv_len - g.q_len + g.t0;  // position of the tile's first token
        const long long limit = (p.causal && row_ok) ? min(kv_len - 1, pos0 + tr) : kv_len - 1;
        const long long tile_limit = p.causal ? min(kv_len - 1, pos0) : kv_len - 1;  // smallest row limit
        float m = -INFINITY, l = 0.f;

        for (int j = 0; j < g.nb; ++j, ++sblk) {
            const uint32_t tS = tmem + lane_off + (sblk & 1u) * 128u;
            ok = __all_sync(0xffffffffu, wait_bar(&b.s_full[sblk & 1u], (sblk >> 1) & 1u, abort_flag, p.status));
            if (!ok) break;
            const long long kbase = (long long)(g.kb0 + j) * 128;
            float alpha = 1.f;
            bool resc = false;
            if (!idle) {  // a warp whose rows are all padding keeps only the barrier protocol and V clearing
                tc_fence_after();
                uint32_t s[128];
                tmem_ld32(tS + 0, s);
                tmem_ld32(tS + 32, s + 32);
                tmem_ld32(tS + 64, s + 64);
                tmem_ld32(tS + 96, s + 96);
                tmem_ld_wait();
                reg_after_wait<128>(s);

                if (kbase + 127 > tile_limit) {  // visible columns of this row: [0, bound)
                    const long long bl = limit - kbase + 1;
                    const int bound = bl < 0 ? 0 : (bl > 128 ? 128 : (int)bl);
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= bound) s[c] = __float_as_uint(-INFINITY);
                }
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
                const float m_use = (m == -INFINITY) ? 0.f : m;
                const uint64_t cs2 = f2_pack(cs, cs);
                const uint64_t nm2 = f2_pack(-m_use, -m_use);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // 32 scores -> 16 packed bf16 P words per chunk
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float p0, p1;
                        f2_unpack(
                            f2_fma(f2_pack(__uint_as_float(s[32 * q + 2 * i]), __uint_as_float(s[32 * q + 2 * i + 1])),
                                   cs2, nm2),
                            p0, p1);
                        p0 = ex2(p0);
                        p1 = ex2(p1);
                        acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
                        w[i] = pack_bf16(p0, p1);
                    }
                    tmem_st16(tS + 16 * q, w);
                }
                {
                    float a0, a1;
                    f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
                    l += a0 + a1;
                }
            }
            if (j > 0) {  // O holds PV_{j-1} once its phase completed; rescale it if the max moved
                ok = __all_sync(0xffffffffu, wait_bar(b.o_full, ocnt & 1u, abort_flag, p.status));
                ++ocnt;
                if (!ok) break;
                tc_fence_after();
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
            }
            if (kbase + 128 > kv_len) {
                // the block runs past the request's keys: clear those V rows (a partial
                // last page holds arbitrary bytes there; pages past it were zero-filled)
                const int iV = kv_base + 2 * j + 1;
                ok = __all_sync(0xffffffffu, wait_bar(&b.kv_full[iV % C::NST], (uint32_t)((iV / C::NST) & 1),
                                                      abort_flag, p.status));
                if (!ok) break;
                if (kbase + row >= kv_len) {
                    const uint32_t vrow = kv_smem + (uint32_t)((iV % C::NST) * C::TILE_BYTES + row * 128);
#pragma unroll
                    for (int pn = 0; pn < C::NPANEL; ++pn)
#pragma unroll
                        for (int c = 0; c < 128; c += 16) st_shared_zero16(vrow + (uint32_t)(pn * C::PANEL_BYTES + c));
                    fence_async_smem();
                }
            }
            tmem_st_wait();
            tc_fence_before();
            bar_arrive(b.p_full);
        }
        if (!ok) break;
        kv_base += 2 * g.nb;

        // ---- epilogue: O -> registers (then release O), / l, store
        ok = __all_sync(0xffffffffu, wait_bar(b.o_full, ocnt & 1u, abort_flag, p.status));
        ++ocnt;
        if (!ok) break;
        tc_fence_after();
        uint32_t o[D];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(tO + 32 * ch, o + 32 * ch);
        tmem_ld_wait();
        reg_after_wait<D>(o);
        tc_fence_before();
        bar_arrive(b.o_empty);
        const float m_use = (m == -INFINITY) ? 0.f : m;
        if (p.n_splits == 1 || g.split < 0) {
            if (!row_ok) continue;
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            uint16_t* dst = p.o + grow * D;
#pragma unroll
            for (int c = 0; c < D; c += 8)
                st_global_v4(dst + c, pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv),
                             pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv),
                             pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv),
                             pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv));
            if (p.lse != nullptr) p.lse[grow] = (l > 0.f) ? (m_use + lg2(l)) * kLn2 : -INFINITY;
        } else if (row_ok) {
            const size_t rec = grow * (size_t)p.n_splits + (size_t)g.split;
            float* po = p.part_o + rec * D;
#pragma unroll
            for (int c = 0; c < D; c += 4) st_global_v4(po + c, o[c], o[c + 1], o[c + 2], o[c + 3]);
            *reinterpret_cast<float2*>(p.part_ml + rec * 2) = make_float2((l > 0.f) ? m_use : -INFINITY, l);
        }
    }
}

// ---------------------------------------------------------------- kernels

template <int D>
__global__ void __launch_bounds__(kPagedThreads, 1) paged_kernel(const __grid_constant__ PagedParams p) {
    using C = PCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    PBars b;
    b.q_full = bars;
    b.q_empty = bars + 2;
    b.kv_full = bars + 4;
    b.kv_empty = bars + 4 + C::NST;
    b.s_full = bars + 4 + 2 * C::NST;
    b.p_full = b.s_full + 2;
    b.o_full = b.p_full + 1;
    b.o_empty = b.o_full + 1;
    b.done = b.o_empty + 1;
    b.uq_full = b.done + 1;
    b.uq_empty = b.uq_full + kQN;
    volatile int* uq = reinterpret_cast<volatile int*>(smem + C::OFF_UQ);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            bar_init(&b.q_full[i], 1);
            bar_init(&b.q_empty[i], 1);
        }
        for (int i = 0; i < kQN; ++i) {
            bar_init(&b.uq_full[i], 1);
            bar_init(&b.uq_empty[i], 5);
        }
        for (int s = 0; s < C::NST; ++s) {
            bar_init(&b.kv_full[s], 1);
            bar_init(&b.kv_empty[s], 1);
        }
        bar_init(&b.s_full[0], 1);
        bar_init(&b.s_full[1], 1);
        bar_init(b.p_full, 128);
        bar_init(b.o_full, 1);
        bar_init(b.o_empty, 128);
        bar_init(b.done, 1);
        *abort_flag = 0;
        bar_init_fence();
    }
    if (warp >= 2) {
        // rows of the Q tile that no load writes (G * T < 128, or fewer tokens
        // in the box) must read as zeros, not stale shared memory
        const uint32_t q0 = smem_u32(smem + C::OFF_Q) + (uint32_t)((threadIdx.x - 64) * (2 * C::TILE_BYTES / 128));
#pragma unroll
        for (int c = 0; c < 2 * C::TILE_BYTES / 128; c += 16) st_shared_zero16(q0 + (uint32_t)c);
        fence_async_smem();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, C::TM_COLS);
        tmem_relinquish();
    }
    griddep_launch_dependents();  // the merge kernel may be scheduled; it waits for this grid
    if (threadIdx.x == 0) *skip = timeout_recorded(p.status) ? 1 : 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (*skip) {  // an earlier launch gave up
        if (warp == 0) tmem_dealloc(tmem, C::TM_COLS);
        return;
    }

    if (warp >= 2) {
        softmax_role<D>(p, smem, b, uq, abort_flag, tmem, warp & 3, lane);
    } else if (warp == 1) {
        if (lane == 0) {
            mma_role<D>(p, smem, b, uq, abort_flag, tmem);
            tc_commit(b.done);  // every issued MMA finishes before tensor memory is released
            drain_wait(b.done, 0, p.status);
        }
        __syncwarp();
    } else {
        producer_role<D>(p, smem, b, uq, abort_flag, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

// Schedule pass (one CTA): the list of units that have work (KV blocks to
// process, or rows to zero when nothing is visible), each entry the unit and
// its request's extent (q_start, q_len, kv_len); its length in sched[1]; the
// fetch counter sched[0] reset to 0.  The list is ordered by work, longest
// first (units with at least kBuckets - 1 blocks share the first bucket), so
// the last units the persistent CTAs take are the shortest.  The H_kv units
// of one (split, tile, request) group have the same work and are listed
// together.  Requests whose offsets or length are out of range are reported
// here, and their clamped extent is what the list carries.
constexpr int kBuckets = 64;
constexpr int kCachedReqs = 2048;

__global__ void __launch_bounds__(1024) paged_schedule_kernel(const PagedParams p) {
    __shared__ int s_qstart[kCachedReqs], s_qlen[kCachedReqs], s_kvlen[kCachedReqs];
    __shared__ int s_bucket[kBuckets];
    __shared__ unsigned long long s_work;
    griddep_launch_dependents();  // the paged kernel may start its prologue now
    const int t = threadIdx.x, lane = t & 31;
    const bool cached = p.B <= kCachedReqs;
    if (t == 0) s_work = 0ull;
    __syncthreads();
    bool bad = false;
    unsigned long long work = 0;  // KV blocks of this thread's requests (one tile each when whole is set)
    for (int r = t; r < p.B; r += 1024) {
        PUnit g;
        request_extent(p, r, g);
        bad |= g.bad;
        if (cached) {
            s_qstart[r] = g.q_start;
            s_qlen[r] = g.q_len;
            s_kvlen[r] = g.kv_len;
        }
        if (p.whole != nullptr && g.q_len > 0) work += (unsigned long long)tile_kv_blocks(p, g.q_len, g.kv_len, min(p.T, g.q_len) - 1);
    }
    if (bad) atomicOr(p.status, 1u << kStatusDeviceData);
    if (t < kBuckets) s_bucket[t] = 0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) work += __shfl_xor_sync(0xffffffffu, work, o);
    if (lane == 0 && work) atomicAdd(&s_work, work);
    __syncthreads();
    // Decode-like launches (one query tile per request): a request whose KV
    // blocks are at most half of a CTA's share of the launch (or one split)
    // runs as one unit -- no partials, no merge -- and only the longer ones
    // are split, so that the work still balances over the CTAs.
    const long long share = (long long)(s_work * (unsigned long long)p.H_kv / (unsigned long long)(2 * p.n_ctas));
    const long long thresh = share > p.split_blocks ? share : p.split_blocks;
    auto is_whole = [&](const PUnit& g) {
        return p.whole != nullptr && g.q_len > 0 && tile_kv_blocks(p, g.q_len, g.kv_len, min(p.T, g.q_len) - 1) <= thresh;
    };
    if (p.whole != nullptr) {
        for (int r = t; r < p.B; r += 1024) {
            PUnit g;
            if (cached) {
                g.q_start = s_qstart[r];
                g.q_len = s_qlen[r];
                g.kv_len = s_kvlen[r];
            } else {
                request_extent(p, r, g);
            }
            p.whole[r] = is_whole(g) ? 1 : 0;
        }
    }
    // group gi -> its first unit gi * H_kv, the request's extent, and its
    // work: KV blocks (0 for a unit that only zeroes rows), -1 for none
    auto group = [&](int gi, PUnit& g) {
        const int r = gi % p.B;
        if (cached) {
            g.q_start = s_qstart[r];
            g.q_len = s_qlen[r];
            g.kv_len = s_kvlen[r];
        } else {
            request_extent(p, r, g);
        }
        unit_tile(p, gi * p.H_kv, g);
        if (is_whole(g)) {  // split 0 only, over all the tile's blocks
            if (g.split > 0) return -1;
            make_whole(p, g);
            return g.nb > 0 ? g.nb : (g.nt > 0 ? 0 : -1);
        }
        if (g.nb > 0) return g.nb;
        return (p.n_splits == 1 && g.nt > 0) ? 0 : -1;
    };
    auto bucket = [](int w) { return w >= kBuckets - 1 ? 0 : kBuckets - 1 - w; };  // longest first
    // Lanes of a warp that hit the same bucket add to it once, through their
    // leader; the returned base plus the lane's rank among them (times H_kv
    // entries per lane) is its place.
    auto reserve = [&](int bk, bool active) {
        const unsigned act = __ballot_sync(0xffffffffu, active);
        const unsigned peers = __match_any_sync(0xffffffffu, active ? bk : -1) & act;
        const int leader = __ffs(peers) - 1;
        int base = 0;
        if (active && lane == leader) base = atomicAdd(&s_bucket[bk], __popc(peers) * p.H_kv);
        base = __shfl_sync(0xffffffffu, base, leader < 0 ? 0 : leader);
        return base + __popc(peers & ((1u << lane) - 1u)) * p.H_kv;
    };
    const int n_groups = p.n_units / p.H_kv;
    const int n_pad = (n_groups + 1023) / 1024 * 1024;  // every lane of a warp runs every round
    for (int gi = t; gi < n_pad; gi += 1024) {
        PUnit g;
        const int w = gi < n_groups ? group(gi, g) : -1;
        reserve(w >= 0 ? bucket(w) : 0, w >= 0);
    }

    __syncthreads();
    if (t < 32) {  // exclusive scan of the 64 bucket counts (two per lane)
        const int a = s_bucket[2 * t], b = s_bucket[2 * t + 1];
        int x = a + b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (t >= o) x += y;
        }
        const int excl = x - a - b;
        s_bucket[2 * t] = excl;
        s_bucket[2 * t + 1] = excl + a;
        if (t == 31) p.sched[1] = x;
    }
    __syncthreads();
    for (int gi = t; gi < n_pad; gi += 1024) {
        PUnit g;
        const int w = gi < n_groups ? group(gi, g) : -1;
        const int pos = reserve(w >= 0 ? bucket(w) : 0, w >= 0);
        const int flag = (w >= 0 && g.split < 0) ? kWholeBit : 0;
        if (w >= 0)
            for (int h = 0; h < p.H_kv; ++h)
                p.sched_list[pos + h] = make_int4((gi * p.H_kv + h) | flag, g.q_start, g.q_len, g.kv_len);
    }
    if (t == 0) p.sched[0] = 0;
}

// One warp per output row (query token, query head): combine the row's
// splits with the (m, l, O) merge, m = max_s m_s, l = sum_s l_s 2^(m_s - m),
// O = sum_s 2^(m_s - m) O_s / l, and write O (bf16) and the LSE.
template <int D>
__global__ void __launch_bounds__(512) paged_merge_kernel(const PagedParams p) {
    constexpr int PER = D / 32;
    static_assert(PER == 4 || PER == 2, "head dim");
    griddep_wait();  // launched early: the partials are complete past this point
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (long long)p.total_q * p.H) return;
    const int tok = (int)(gw / p.H);
    int r = tok;
    if (p.cu_q != nullptr) {  // the last request whose first token is <= tok
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.cu_q + mid) <= tok)
                lo = mid;
            else
                hi = mid - 1;
        }
        r = lo;
    }
    PUnit g;
    request_extent(p, r, g);
    const int t = tok - g.q_start;
    if (t < 0 || t >= g.q_len) return;  // token not owned by a valid request (reported by the main kernel)
    if (p.whole != nullptr && __ldg(p.whole + r)) return;  // written by its unit
    const int t0 = (t / p.T) * p.T;
    const int nb = tile_kv_blocks(p, g.q_len, g.kv_len, min(t0 + p.T, g.q_len) - 1);
    const int ns = (nb + p.split_blocks - 1) / p.split_blocks;
    const size_t rec0 = (size_t)gw * p.n_splits;

    // lane s holds split s's (m, l) for s < 32 (more splits: further rounds)
    float m = -INFINITY;
    for (int s = lane; s < ns; s += 32) m = fmaxf(m, p.part_ml[(rec0 + s) * 2]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    float acc[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c) acc[c] = 0.f;
    if (m != -INFINITY) {
        for (int s0 = 0; s0 < ns; s0 += 32) {
            float w_mine = 0.f;  // weight 2^(m_s - m) of this lane's split
            if (s0 + lane < ns) {
                const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + (rec0 + s0 + lane) * 2);
                w_mine = ex2(ml.x - m);
                l += ml.y * w_mine;
            }
            const int cnt = min(32, ns - s0);
            // lane owns PER consecutive dims of O: one 16-byte (d = 128) or
            // 8-byte (d = 64) load per split, eight loads in flight
            for (int s = 0; s < cnt; s += 8) {
                float w[8];
                float v[8][PER];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    w[i] = __shfl_sync(0xffffffffu, w_mine, (s + i) & 31);
                    const bool in = s + i < cnt;
                    const float* src = p.part_o + (rec0 + s0 + s + (in ? i : 0)) * D + lane * PER;
                    if (PER == 4) {
                        const float4 x = in ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[i][0] = x.x;
                        v[i][1] = x.y;
                        v[i][PER > 2 ? 2 : 0] = x.z;
                        v[i][PER > 3 ? 3 : 0] = x.w;
                    } else {
                        const float2 x = in ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
                        v[i][0] = x.x;
                        v[i][1] = x.y;
                    }
                    if (!in) w[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int c = 0; c < PER; ++c) acc[c] = fmaf(w[i], v[i][c], acc[c]);
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    uint16_t* dst = p.o + (size_t)gw * D + lane * PER;
    if (PER == 4)
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(acc[0] * inv, acc[1] * inv),
                                                    pack_bf16(acc[2] * inv, acc[3] * inv));
    else
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
    if (lane == 0 && p.lse != nullptr) p.lse[gw] = (l > 0.f) ? (m + lg2(l)) * kLn2 : -INFINITY;
}

template <int D>
cudaError_t launch_d(const PagedParams& p, int grid, cudaStream_t stream) {
    using C = PCfg<D>;
    cudaError_t e =
        cudaFuncSetAttribute(paged_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    paged_schedule_kernel<<<1, 1024, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // programmatic dependent launches: the paged kernel's prologue overlaps
    // the schedule pass and its producer waits for the pass (griddepcontrol.wait)
    // before reading the list; the merge kernel is scheduled early and waits
    // for the paged kernel to complete
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kPagedThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, paged_kernel<D>, p);
    if (e != cudaSuccess || p.n_splits == 1) return e;
    const long long warps = (long long)p.total_q * p.H;
    cfg.gridDim = dim3((unsigned)((warps + 15) / 16));
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, paged_merge_kernel<D>, p);
}

}  // namespace

PagedPlan paged_plan(int total_q, int max_q_len, int B, int H, int H_kv, int d, int page_size, int max_pages) {
    PagedPlan pl{};
    pl.G = H / H_kv;
    pl.T = 128 / pl.G;
    if (pl.T > max_q_len) pl.T = max_q_len;
    if (pl.T < 1) pl.T = 1;
    pl.n_qt = (max_q_len + pl.T - 1) / pl.T;
    const long long kv_blocks = ((long long)max_pages * page_size + 127) / 128;
    const long long base = (long long)B * H_kv * pl.n_qt;
    // Decode-like launches (one query tile per request) split every request
    // into runs of 8 KV blocks so lengths that differ by 16x still balance
    // over the SMs; multi-tile launches split only when there are too few
    // units to fill the GPU.
    long long sb = 8;
    if (pl.n_qt > 1) {
        const long long want = (1024 + base - 1) / base;  // splits per unit wanted
        sb = (kv_blocks + want - 1) / want;
        if (sb < 8) sb = 8;
    }
    if (sb > kv_blocks) sb = kv_blocks;
    if (sb < 1) sb = 1;
    pl.split_blocks = (int)sb;
    pl.n_splits = (int)((kv_blocks + sb - 1) / sb);
    pl.n_units = base * pl.n_splits;
    // header (fetch counter, list length), the unit list, then the partials
    pl.list_offset = 256;
    pl.workspace_bytes = 256 + ((size_t)pl.n_units * 16 + 255) / 256 * 256;
    if (pl.n_splits > 1) {
        const size_t recs = (size_t)total_q * H * pl.n_splits;
        pl.part_o_bytes = recs * d * sizeof(float);
        pl.part_ml_bytes = recs * 2 * sizeof(float);
        pl.part_o_offset = pl.workspace_bytes;
        pl.workspace_bytes += (pl.part_o_bytes + 255) / 256 * 256;
        pl.part_ml_offset = pl.workspace_bytes;
        pl.workspace_bytes += pl.part_ml_bytes;
        // decode-like launches: per-request flags for requests run unsplit
        if (pl.n_qt == 1 && pl.n_units < (1LL << 30)) {
            pl.workspace_bytes = (pl.workspace_bytes + 255) / 256 * 256;
            pl.whole_offset = pl.workspace_bytes;
            pl.workspace_bytes += (size_t)B * sizeof(int);
        }
    }
    return pl;
}

int paged_smem_bytes(int d) {
    if (d == 128) return PCfg<128>::SMEM_BYTES;
    if (d == 64) return PCfg<64>::SMEM_BYTES;
    return -1;
}

cudaError_t launch_paged(int d, const PagedParams& p, int grid, cudaStream_t stream) {
    if (d == 128) return launch_d<128>(p, grid, stream);
    if (d == 64) return launch_d<64>(p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
