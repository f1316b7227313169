// Chunked prefill attention over the paged KV cache on the 5th-generation
// tensor cores (tcgen05 MMAs, accumulators in tensor memory).
//
// "KV cache, PagedAttention and FlashAttention" (Problem 4 and the
// FlashAttention discussion): a chunk of T new tokens of sequence b, already
// appended at positions C-T .. C-1 of its cache (C = context_lens[b]),
// attends causally to positions 0 .. C-T+i of its own cache through the
// block table.  The query rows of one KV head g are (token i, head h of g's
// group), row r = i * G + h, so the G heads that share a KV head share every
// key and value tile: the grouped-query structure becomes the M dimension of
// the two products S = Q K^T and O = P V.
//
// Design (one persistent CTA per SM, warp-specialised):
//   * a tile is 128 query rows of one (sequence, KV head); the tile list is
//     sequence-major, then KV head, then row tile, so the CTAs running at one
//     time share a few sequences' K/V in L2.  CTA c takes tiles c, c + grid,
//     ...; every warp walks the list itself from the chunk lengths (a window
//     of 32 sequences held in registers), so no role hands tiles to another.
//   * warp 4 streams Q (one 3-D TMA box per 64 columns) and the K tiles of
//     128 keys (8 blocks of 16 tokens, one 2-D TMA box per block and 64
//     columns) into a two-stage ring; warp 5 streams the V tiles likewise.
//     A missing block or an out-of-range block id loads a box past the end of
//     the pool (zero filled) and is masked out of the scores.
//   * warp 6 issues the MMAs from one thread: S = Q K^T for step j into one
//     of two S accumulators in tensor memory (128 columns each), then
//     O += P V for step j-1 (P from shared memory), so the tensor cores
//     compute the next scores while the softmax warps work on the current.
//   * warps 0-3 own one query row each (row = TMEM lane): they read the row's
//     128 scores, mask by position and block validity, and keep the online
//     softmax in the exp2 domain with a lazily updated reference maximum: the
//     accumulator O is rescaled (read, scaled and written back in tensor
//     memory) only when a row's maximum grows by more than 2^8, so P stays
//     at most 256 and almost every step skips the rescale.  P is rounded to
//     bf16 for the MMA and the row sum l adds the rounded values, so the
//     result is exactly a convex combination of the V rows with the weights
//     the MMA used.  After the tile's last step they read O, divide by l and
//     store bf16.
// Every mbarrier wait is bounded; on a timeout the CTA records
// PKV_DEVERR_TIMEOUT, every role stops, the MMA and copy pipes are drained
// (bounded) and the tensor memory is released before the CTA exits.
#include <algorithm>
#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kRows = 128;               // query rows per tile (= TMEM lanes)
constexpr int kKeys = 128;               // keys per step
constexpr int kStepBlocks = kKeys / kBlockSize;
constexpr int kSoftmaxWarps = 4;
constexpr int kKWarp = 4, kVWarp = 5, kMmaWarp = 6;
constexpr int kThreads = 7 * 32;
constexpr float kRescaleSlack = 8.0f;    // log2 of the largest P value allowed before O is rescaled
constexpr uint32_t kTmemCols = 512;      // S0 at 0, S1 at 128, O at 256
constexpr uint32_t kColO = 256;
constexpr uint32_t kHalf = 128 * 128;    // bytes of one 64-column half of a 128-row tile

struct Args {
    const int32_t *qo_indptr;  // [batch + 1]
    const int32_t *block_tables;
    int W;
    const int32_t *context_lens;
    int batch, n_q, n_kv;
    int64_t num_blocks;
    int64_t n_rows;            // rows of q and out: stores past them are skipped (an inconsistent indptr)
    int oob_row;               // a K/V row index past the end of the pool (zero-filled box)
    float qscale;              // scale * log2(e)
    __nv_bfloat16 *out;        // [rows][n_q][D]
    unsigned *err;
};

template <int D>
struct Layout {
    static constexpr uint32_t QT = kRows * D * 2;        // one Q tile
    static constexpr uint32_t KT = kKeys * D * 2;        // one K (or V) step
    static constexpr uint32_t PT = kRows * kKeys * 2;    // P, bf16
    static constexpr uint32_t kQ = 0;                    // 2 Q buffers
    static constexpr uint32_t kK = kQ + 2 * QT;          // 2 K stages
    static constexpr uint32_t kV = kK + 2 * KT;          // 2 V stages
    static constexpr uint32_t kP = kV + 2 * KT;
    static constexpr uint32_t kBar = kP + PT;
    enum { Q_FULL = 0, Q_FREE = 2, K_FULL = 4, K_EMPTY = 6, V_FULL = 8, V_EMPTY = 10, S_FULL = 12, S_FREE = 14,
           P_FULL = 16, O_DONE = 17, DRAIN = 18, NBARS = 19 };
    static constexpr uint32_t kTmemSlot = kBar + NBARS * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr size_t bytes = 1024 + kEnd;
};

// ------------------------------------------------------------- tcgen05 PTX

// Shared-memory matrix descriptor: 128-byte swizzled canonical layout.  For a
// K-major operand `sbo` is the stride between 8-row groups (1024 B) and the
// leading offset is unused; for an MN-major operand `lbo` is the stride
// between 64-element chunks of the M/N dimension and `sbo` the stride
// between 8-row groups of the K dimension.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: bf16 A and B, f32 accumulator, M x N,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, int b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}

// Arrive once on `bar` when every tcgen05 MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive columns of this warp's 32 TMEM lanes, one lane per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
                 "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                   "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
                   "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
                   "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled
// tile of 128-byte rows starting on a 1024-byte boundary.
__device__ __forceinline__ uint32_t swz_off(int row, int chunk)
{
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ------------------------------------------------------------- tile walk

struct Tile {
    int b, g, rt0;  // sequence, KV head, first local row
    int R;          // rows of (b, g): T * G
    int row0, T, C; // first query token row of b, chunk length, context length (clamped)
    int n_blocks, n_steps;
    bool bad_ctx;   // context length out of range (recorded once per tile by the softmax warps)
};

// A window of 32 sequences held one per lane: each warp walks the tile list
// itself, with the same arithmetic, so every role sees the same tiles.
struct Walker {
    int wb = 0;           // first sequence of the window
    long long wbase = 0;  // tiles before sequence wb
    long long incl = 0, tot = 0;
    int n = 0, row0 = 0, T = 0, C = 0;
};

template <int G>
__device__ __forceinline__ void load_window(Walker &w, const Args &a, int lane)
{
    const int bl = w.wb + lane;
    w.row0 = w.T = w.C = 0;
    long long n = 0;
    if (bl < a.batch) {
        w.row0 = a.qo_indptr[bl];
        w.T = a.qo_indptr[bl + 1] - w.row0;
        w.C = a.context_lens[bl];
        if (w.T > 0) n = (long long)a.n_kv * (((long long)w.T * G + kRows - 1) / kRows);
    }
    long long x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    w.n = (int)n;
    w.incl = x;
    w.tot = __shfl_sync(kFull, x, 31);
}

// Tile x of the list; false past its end.  Warp-wide, uniform result.
template <int G>
__device__ __forceinline__ bool find_tile(Walker &w, const Args &a, long long x, Tile &t, int lane)
{
    while (x >= w.wbase + w.tot) {
        if (w.wb + 32 >= a.batch) return false;
        w.wbase += w.tot;
        w.wb += 32;
        load_window<G>(w, a, lane);
    }
    const unsigned hit = __ballot_sync(kFull, w.wbase + w.incl > x);
    const int l = __ffs(hit) - 1;
    const long long before = __shfl_sync(kFull, w.incl - w.n, l);
    const int n = __shfl_sync(kFull, w.n, l);
    t.b = w.wb + l;
    t.row0 = __shfl_sync(kFull, w.row0, l);
    t.T = __shfl_sync(kFull, w.T, l);
    int C = __shfl_sync(kFull, w.C, l);
    const int per_head = n / a.n_kv;
    const int within = (int)(x - w.wbase - before);
    t.g = within / per_head;
    t.rt0 = (within % per_head) * kRows;
    t.R = t.T * G;
    const int cap = a.W * kBlockSize;
    t.bad_ctx = C < t.T || C > cap;
    if (t.bad_ctx) C = max(t.T, min(C, cap));
    t.C = C;
    if (C > cap) {  // a chunk longer than the whole table: nothing sensible to attend to
        t.n_blocks = t.n_steps = 0;
        return true;
    }
    const int last_row = min(t.R, t.rt0 + kRows) - 1;
    t.n_blocks = (C - t.T + last_row / G) / kBlockSize + 1;
    t.n_steps = (t.n_blocks + kStepBlocks - 1) / kStepBlocks;
    return true;
}

__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity)
{
    return __all_sync(kFull, mbar_wait_bounded(bar, parity));
}

// ------------------------------------------------------------- the kernel

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, Args a)
{
    using L = Layout<D>;
    constexpr int NH = D / 64 > 0 ? D / 64 : 1;  // 64-column halves of a row
    extern __shared__ __align__(1024) uint8_t tc_smem[];
    uint8_t *sm = tc_smem + ((1024u - (smem_u32(tc_smem) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kBar);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kAbort);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        for (int i = 0; i < L::NBARS; ++i) {
            const bool by_warps = i == L::S_FREE || i == L::S_FREE + 1 || i == L::P_FULL;
            mbar_init(&bar[i], by_warps ? kSoftmaxWarps : 1);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(sm + L::kTmemSlot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + L::kTmemSlot);
    griddep_wait();  // queries, tables and the appended chunk may come from the previous kernel
    griddep_launch_dependents();

    auto set_abort = [&]() {
        if (lane == 0) {
            atomicOr(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    };

    Walker wk;
    load_window<G>(wk, a, lane);

    if (warp == kKWarp || warp == kVWarp) {
        // ---------------------------------------------------------- producers
        const bool is_k = warp == kKWarp;
        const CUtensorMap *map = is_k ? &tm_k : &tm_v;
        const uint32_t ring = is_k ? L::kK : L::kV;
        uint64_t *full = &bar[is_k ? L::K_FULL : L::V_FULL];
        uint64_t *empty = &bar[is_k ? L::K_EMPTY : L::V_EMPTY];
        const uint64_t policy = l2_policy_evict_normal();
        int gs = 0, qi = 0;
        bool ok = true;
        for (long long x = blockIdx.x; ok; x += gridDim.x) {
            Tile t;
            if (!find_tile<G>(wk, a, x, t, lane)) break;
            if (t.n_steps == 0) continue;
            if (*abort_flag) break;
            if (is_k) {  // this tile's queries into Q buffer qi & 1
                const int qb = qi & 1;
                if (qi >= 2 && !(ok = wait_all(&bar[L::Q_FREE + qb], ((qi >> 1) + 1) & 1))) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar[L::Q_FULL + qb], L::QT);
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        tma_load_3d(sm + L::kQ + qb * L::QT + h * kHalf, &tm_q, 64 * h, t.g * G,
                                    t.row0 + t.rt0 / G, &bar[L::Q_FULL + qb], policy);
                }
                ++qi;
            }
            const int32_t *trow = a.block_tables + (int64_t)t.b * a.W;
            for (int s = 0; s < t.n_steps; ++s, ++gs) {
                const int st = gs & 1;
                if (gs >= 2 && !(ok = wait_all(&empty[st], ((gs >> 1) + 1) & 1))) break;
                const int blk = s * kStepBlocks + lane;
                bool valid = false;
                int phys = -1;
                if (lane < kStepBlocks && blk < t.n_blocks) {
                    phys = trow[blk];
                    valid = phys >= 0 && phys < a.num_blocks;
                    if (!valid && is_k) atomicOr(a.err, PKV_DEVERR_BLOCK_RANGE);
                }
                if (lane == 0) mbar_arrive_expect_tx(&full[st], L::KT);
                __syncwarp();
                if (lane < kStepBlocks) {
                    const int y = valid ? (int)((phys * (int64_t)a.n_kv + t.g) * kBlockSize) : a.oob_row;
                    uint8_t *dst = sm + ring + st * L::KT + lane * (kBlockSize * 128);
#pragma unroll
                    for (int h = 0; h < NH; ++h) tma_load_2d(dst + h * kHalf, map, 64 * h, y, &full[st], policy);
                }
            }
        }
        // copies still in flight (after an abort) land before the CTA exits
        for (int st = 0; st < 2 && gs - 1 - st >= 0; ++st) {
            const int g2 = gs - 1 - st;
            mbar_wait_bounded(&full[g2 & 1], (g2 >> 1) & 1);
        }
        if (is_k && qi > 0) mbar_wait_bounded(&bar[L::Q_FULL + ((qi - 1) & 1)], ((qi - 1) >> 1) & 1);
        if (is_k && qi > 1) mbar_wait_bounded(&bar[L::Q_FULL + ((qi - 2) & 1)], ((qi - 2) >> 1) & 1);
        if (!ok) set_abort();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issue
        constexpr uint32_t idesc_qk = mma_idesc(kRows, kKeys, 0);
        constexpr uint32_t idesc_pv = mma_idesc(kRows, D, 1);
        const uint32_t base = smem_u32(sm);
        int gs = 0, qi = 0;
        int pv_gs = -1;
        bool pv_acc = false, ok = true;
        auto issue_pv = [&](int g2, bool acc) -> bool {
            if (!wait_all(&bar[L::P_FULL], g2 & 1)) return false;
            if (!wait_all(&bar[L::V_FULL + (g2 & 1)], (g2 >> 1) & 1)) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t pb = base + L::kP, vb = base + L::kV + (g2 & 1) * L::KT;
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk) {
                    const uint64_t ad = smem_desc(pb + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(vb + kk * 2048, kHalf, 1024);
                    umma(tmem + kColO, ad, bd, idesc_pv, (acc || kk > 0) ? 1u : 0u);
                }
                umma_commit(&bar[L::O_DONE]);
                umma_commit(&bar[L::V_EMPTY + (g2 & 1)]);
            }
            __syncwarp();
            return true;
        };
        for (long long x = blockIdx.x; ok; x += gridDim.x) {
            Tile t;
            if (!find_tile<G>(wk, a, x, t, lane)) break;
            if (t.n_steps == 0) continue;
            if (*abort_flag) break;
            const int qb = qi & 1;
            if (!(ok = wait_all(&bar[L::Q_FULL + qb], (qi >> 1) & 1))) break;
            for (int s = 0; s < t.n_steps && ok; ++s, ++gs) {
                const int st = gs & 1;
                if (!(ok = wait_all(&bar[L::K_FULL + st], (gs >> 1) & 1))) break;
                if (gs >= 2 && !(ok = wait_all(&bar[L::S_FREE + st], ((gs >> 1) + 1) & 1))) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t qbase = base + L::kQ + qb * L::QT, kbase = base + L::kK + st * L::KT;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                        umma(tmem + st * kKeys, smem_desc(qbase + off, 16, 1024), smem_desc(kbase + off, 16, 1024),
                             idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&bar[L::S_FULL + st]);
                    umma_commit(&bar[L::K_EMPTY + st]);
                    if (s == t.n_steps - 1) umma_commit(&bar[L::Q_FREE + qb]);
                }
                __syncwarp();
                if (pv_gs >= 0 && !(ok = issue_pv(pv_gs, pv_acc))) break;
                pv_gs = gs;
                pv_acc = s > 0;
            }
            ++qi;
        }
        if (ok && pv_gs >= 0) ok = issue_pv(pv_gs, pv_acc);
        // every MMA issued so far has completed before the tensor memory is released
        if (lane == 0) umma_commit(&bar[L::DRAIN]);
        __syncwarp();
        mbar_wait_bounded(&bar[L::DRAIN], 0);
        if (!ok) set_abort();
    } else {
        // ---------------------------------------------------------- softmax
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        uint8_t *prow = sm + L::kP;
        int gs = 0;
        bool ok = true;
        for (long long x = blockIdx.x; ok; x += gridDim.x) {
            Tile t;
            if (!find_tile<G>(wk, a, x, t, lane)) break;
            if (t.bad_ctx && tid == 0 && t.rt0 == 0 && t.g == 0) atomicOr(a.err, PKV_DEVERR_CTX_RANGE);
            if (t.n_steps == 0) continue;
            if (*abort_flag) break;
            const int r = t.rt0 + tid;
            const int64_t orow_i = (int64_t)t.row0 + min(r, t.R - 1) / G;  // this row's query token
            const bool in_out = orow_i >= 0 && orow_i < a.n_rows;
            if (r < t.R && !in_out) atomicOr(a.err, PKV_DEVERR_CTX_RANGE);
            const bool live = r < t.R && in_out;
            const int pos = t.C - t.T + min(r, t.R - 1) / G;  // this row's position; it sees keys 0 .. pos
            float mref = -INFINITY, l = 0.0f;
            // block ids of the next step (lanes 0..7), read one step ahead: the same
            // validity test as the producers, so a masked block is exactly a skipped one
            const int32_t *trow = a.block_tables + (int64_t)t.b * a.W;
            int nxt = lane < kStepBlocks && lane < t.n_blocks ? trow[lane] : -1;
            for (int s = 0; s < t.n_steps; ++s, ++gs) {
                const int cur = nxt;
                const int nb = (s + 1) * kStepBlocks + lane;
                if (s + 1 < t.n_steps) nxt = lane < kStepBlocks && nb < t.n_blocks ? trow[nb] : -1;
                const uint32_t mask = __ballot_sync(kFull, cur >= 0 && cur < a.num_blocks) & ((1u << kStepBlocks) - 1);
                const int sb = gs & 1;
                if (!(ok = wait_all(&bar[L::S_FULL + sb], (gs >> 1) & 1))) break;
                tc_fence_after();
                uint32_t sr[kKeys];
#pragma unroll
                for (int c = 0; c < kKeys / 32; ++c) tmem_ld32(tmem + lane_off + sb * kKeys + 32 * c, sr + 32 * c);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[L::S_FREE + sb]);

                const int key0 = s * kKeys;
                float bm = -INFINITY;
                if (mask == (1u << kStepBlocks) - 1 && key0 + kKeys - 1 <= pos) {
#pragma unroll
                    for (int k = 0; k < kKeys; ++k) bm = fmaxf(bm, __uint_as_float(sr[k]));
                } else {
#pragma unroll
                    for (int k = 0; k < kKeys; ++k) {
                        const bool vis = ((mask >> (k / kBlockSize)) & 1u) && key0 + k <= pos;
                        if (!vis) sr[k] = __float_as_uint(-INFINITY);
                        bm = fmaxf(bm, __uint_as_float(sr[k]));
                    }
                }
                const float bms = bm * a.qscale;
                const bool resc = bms > mref + kRescaleSlack;
                float alpha = 1.0f;
                if (resc) {
                    alpha = ex2(mref - bms);  // 0 when mref is -inf
                    mref = bms;
                    l *= alpha;
                }
                const float nm = mref == -INFINITY ? 0.0f : -mref;
                uint32_t pk[kKeys / 2];
#pragma unroll
                for (int i = 0; i < kKeys / 2; ++i) {
                    const float p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), a.qscale, nm));
                    const float p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), a.qscale, nm));
                    pk[i] = pack_bf16x2(p0, p1);
                    l += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xffff0000u);
                }
                if (s > 0) {  // the previous step's O += P V has finished: P is free, O is current
                    if (!(ok = wait_all(&bar[L::O_DONE], (gs - 1) & 1))) break;
                    tc_fence_after();
                    if (__any_sync(kFull, resc)) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tmem + lane_off + kColO + 32 * c, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(tmem + lane_off + kColO + 32 * c, o);
                        }
                        tmem_wait_st();
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t *v = pk + 32 * h + 4 * c;
                        *reinterpret_cast<uint4 *>(prow + h * kHalf + swz_off(tid, c)) =
                            make_uint4(v[0], v[1], v[2], v[3]);
                    }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[L::P_FULL]);
            }
            if (!ok) break;
            // epilogue: O / l for this tile's rows
            if (!(ok = wait_all(&bar[L::O_DONE], (gs - 1) & 1))) break;
            tc_fence_after();
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            __nv_bfloat16 *orow = a.out + ((in_out ? orow_i : 0) * a.n_q + t.g * G + min(r, t.R - 1) % G) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + kColO + 32 * c, o);
                tmem_wait_ld();
                if (live) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + 32 * c + 8 * q4) = w;
                    }
                }
            }
            tc_fence_before();
        }
        if (!ok) set_abort();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <int D, int G>
pkv_status launch(pkv_pool *pool, const void *q, int64_t n_rows, int n_q, const Args &a, cudaStream_t s)
{
    using L = Layout<D>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(prefill_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)L::bytes);
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "prefill kernel attributes");
    CUtensorMap tm_q;
    pkv_status st = make_q_map(&tm_q, q, n_rows, n_q, D, G, kRows / G);
    if (st != PKV_OK) return st;
    // an upper bound on the tiles: every sequence may end with a partial row tile
    const int64_t tiles = ((n_rows * G + kRows - 1) / kRows + a.batch) * a.n_kv;
    const int grid = (int)std::min<int64_t>(tiles, std::max(1, pool->num_sms));
    LaunchScope ls(pool, kDecode, s);
    cudaError_t e = launch_pdl(prefill_tc_kernel<D, G>, dim3(grid), dim3(kThreads), L::bytes, s, tm_q, pool->tm_k,
                               pool->tm_v, a);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return PKV_OK;
}

template <int D>
pkv_status dispatch(pkv_pool *pool, const void *q, int64_t n_rows, int n_q, int G, const Args &a, cudaStream_t s)
{
    switch (G) {
    case 1: return launch<D, 1>(pool, q, n_rows, n_q, a, s);
    case 2: return launch<D, 2>(pool, q, n_rows, n_q, a, s);
    case 4: return launch<D, 4>(pool, q, n_rows, n_q, a, s);
    case 8: return launch<D, 8>(pool, q, n_rows, n_q, a, s);
    }
    return fail(PKV_EUNSUPPORTED, "prefill: group size %d unsupported (1, 2, 4 or 8)", G);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_prefill_attention(pkv_pool *pool, const void *q, int64_t n_rows, int32_t n_q,
                                              const int32_t *qo_indptr, const int32_t *block_tables,
                                              int32_t max_blocks_per_seq, const int32_t *context_lens,
                                              int32_t batch, float scale, void *out, void *stream)
{
    pkv_status st = check_step_args(pool, "paged_prefill_attention", n_q, max_blocks_per_seq, batch, scale);
    if (st != PKV_OK || batch == 0 || n_rows == 0) return st;
    if (n_rows < 0) return fail(PKV_EINVAL, "paged_prefill_attention: n_rows < 0");
    if (n_rows > INT32_MAX) return fail(PKV_EUNSUPPORTED, "paged_prefill_attention: more than 2^31 query rows");
    if (pool->dtype != PKV_BF16) return fail(PKV_EUNSUPPORTED, "paged_prefill_attention: bf16 pools only");
    if (!q || !qo_indptr || !block_tables || !context_lens || !out)
        return fail(PKV_EINVAL, "paged_prefill_attention: NULL device pointer");
    if (((uintptr_t)q | (uintptr_t)out) & 15u)
        return fail(PKV_EINVAL, "paged_prefill_attention: q and out must be 16-byte aligned");
    if (((uintptr_t)qo_indptr | (uintptr_t)block_tables | (uintptr_t)context_lens) & 3u)
        return fail(PKV_EINVAL, "paged_prefill_attention: indptr, tables and lengths must be 4-byte aligned");
    Args a;
    a.qo_indptr = qo_indptr;
    a.block_tables = block_tables;
    a.W = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.batch = batch;
    a.n_q = n_q;
    a.n_kv = pool->n_kv;
    a.num_blocks = pool->num_blocks;
    a.n_rows = n_rows;
    a.oob_row = (int)(pool->num_blocks * pool->n_kv * kBlockSize);
    a.qscale = scale * kLog2e;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = pool->err;
    const int G = n_q / pool->n_kv;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return pool->d_head == 128 ? dispatch<128>(pool, q, n_rows, n_q, G, a, s)
                               : dispatch<64>(pool, q, n_rows, n_q, G, a, s);
}
