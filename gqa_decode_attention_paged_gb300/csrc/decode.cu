// Paged GQA decode attention: one new query token per sequence against its
// cached keys and values, read through the sequence's block table.
//
// What is computed ("The KV Cache from First Principles", "Implementation";
// "KV cache, PagedAttention and FlashAttention", Problems 4 and 5):
//   out[b][h] = sum_p softmax_p(scale * q[b][h] . K[p][g]) V[p][g],
//   g = h / (n_q / n_kv), p < context_len[b], K/V of position p in block
//   block_table[b][p / 16] at offset p % 16.
//
// How:
//   * Work list.  The (sequence, KV head, block) items of the whole batch form
//     one stream ordered by sequence, head, block.  It is cut into equal
//     slices, one per warp of a persistent grid (#SMs x resident CTAs x warps
//     per CTA), so every warp gets the same number of blocks whatever the
//     length mix, and long sequences are split across warps and SMs ("KV
//     cache, PagedAttention and FlashAttention", Problem 5, "Serving note";
//     "Memory Management in LLM Serving Systems", FlashAttention-2:
//     parallelise over the sequence dimension).  Block counts per sequence
//     come from an in-kernel prefix sum over context_lens, so the host never
//     reads lengths and the call never synchronises.
//   * Warps are independent: after the prologue there is no CTA barrier.  A
//     warp's slice meets one or more (sequence, head) runs; each meeting is a
//     "piece".  The warp owns a ring of shared-memory stages that its lane 0
//     fills with tiled TMA copies (cp.async.bulk.tensor, swizzled,
//     evict-first) of a block's K and V tiles, completing on an mbarrier (a
//     4-bit pool's (block, head) entry of key codes, value codes and value
//     parameters arrives as one bulk copy); block-table entries are fetched a
//     segment ahead with one coalesced load.  Every wait is bounded.
//   * All G query heads of the group are served from one read of each tile
//     ("Memory Management in LLM Serving Systems", FlashAttention: query
//     heads sharing a KV head cut KV reads by the group factor): they are the
//     N dimension of 16x8x16 tensor-core MMAs, S^T = K Q^T then O^T += V^T P^T.
//   * Online softmax in fp32 with exp2 (scores pre-scaled by scale*log2 e):
//     per head a reference maximum and a running sum; weights are taken
//     against the reference, which is raised (and the sum and accumulator
//     rescaled) only when a score passes it by more than a small slack, and
//     1/l is applied once at the end (Problem 5's recurrence;
//     FlashAttention-2's deferred normalisation).
//   * Piece end: a piece that is its whole (sequence, head) writes bf16 `out`.
//     Otherwise it stores (m, l, O) in the workspace, and merge_kernel,
//     launched right behind as a programmatic dependent, combines each
//     (sequence, head)'s pieces in slice order by log-sum-exp: M = max m_p,
//     L = sum 2^(m_p-M) l_p, out = sum 2^(m_p-M) O_p / L.  No warp waits for
//     another, and the result does not depend on which warp finished first.
//   * FP8 KV: tiles are E4M3, converted to f16 pairs in registers for f16
//     MMAs; the K scale is folded into the score scale and the V scale into
//     the final normalisation.
//   * 4-bit KV: codes enter f16 MMAs as 1024 + c (see i4_lo), the keys'
//     per-channel scales are folded into q, and each value row's scale and
//     zero point into P and a per-head correction at the piece end.
#include <algorithm>
#include <type_traits>
#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {

constexpr int kMinBlocksPerWarp = 8;

struct DecodeArgs {
    int64_t num_blocks;
    int n_kv, n_q;
    const __nv_bfloat16 *q;
    const int32_t *block_tables;  // dense [batch][W], or with indptr the CSR page list
    int W;
    const int32_t *indptr;        // CSR form: sequence b owns block_tables[indptr[b] .. indptr[b+1]); null: dense
    int64_t n_indices;            // CSR form: entries of block_tables
    const int32_t *context_lens;
    int batch;
    float qscale;          // scale * log2(e)
    const float *scales;   // FP8: [2 * n_kv] (k then v)
    const float *k_params; // 4-bit: [2][n_kv][D] key scales, then zero points
    const uint8_t *i4_entries;  // 4-bit: the pool's [num_blocks][n_kv] (block, KV head) entries
    __nv_bfloat16 *out;
    float2 *ws_ml;         // workspace [slots][G] (max in log2 units, sum)
    float *ws_o;           // workspace [slots][G][D], unnormalised
    int slice_blocks;      // blocks per slice; 0 = ceil(total / all warps)
    unsigned *err;
    // fused step only: the token at position context_len-1 of each sequence,
    // [batch][n_kv][D] bf16, and the pool arrays it is appended to
    const __nv_bfloat16 *k_new, *v_new;
    uint8_t *k_pool;  // the pool's first (block, KV head) entry
    // cascade decode only: the first skip_blocks table entries of every
    // sequence are a shared prefix whose attention comes from n_pre chunk
    // partials (see MergeArgs); the kernel covers the blocks after it
    int skip_blocks, n_pre;
    int64_t pre_base;
};

// KV storage types the decode kernel is instantiated for (pkv_dtype values)
constexpr int kKvBf16 = 0, kKvFp8 = 1, kKvInt4 = 2;

// Shared-memory geometry of one (block, KV head) stage.  bf16 and FP8: the
// pool entry's 32 rows (16 key rows, then 16 value rows) as NREG TMA boxes of
// 32 rows x BOXB bytes lay them out, one box per BOXB-byte column range
// (128-byte boxes; 64 bytes for FP8 with d_head 64), each swizzled within its
// own region: column range r's key rows at r x CSTRIDE, its value rows RGN
// after them.  4-bit: the pool's entry as one bulk copy lays it out,
// unswizzled: 16 key rows of d/2 code bytes, 16 value rows, then the value
// rows' 16 (scale, zero point) pairs at PARAMS.
template <int D, int KV>
struct Geo {
    static constexpr bool FP8 = KV == kKvFp8, I4 = KV == kKvInt4;
    static constexpr int E = FP8 || I4 ? 1 : 2;           // bytes per stored element (a byte of two codes)
    static constexpr int ROWB = I4 ? D / 2 : D * E;       // bytes of one token row
    static constexpr int BOXB = ROWB > 128 ? 128 : ROWB;  // bytes of one box row
    static constexpr int NREG = ROWB / BOXB;              // boxes per tile
    static constexpr int RGN = kBlockSize * BOXB;         // bytes per box
    static constexpr int TILE = NREG * RGN;               // K tile (or V tile) bytes
    static constexpr int CSTRIDE = 2 * RGN;               // between column ranges (key then value rows)
    static constexpr int VOFF = RGN;                      // value rows after their column range's key rows
    static constexpr int PARAMS = 2 * TILE;               // 4-bit: offset of the value parameters
    static constexpr int STAGE = 2 * TILE + (I4 ? kBlockSize * 8 : 0);
    static_assert(!I4 || STAGE == i4_entry_bytes(D), "a 4-bit stage holds exactly one pool entry");
    static constexpr int BOX_ELEMS = BOXB / E;
};

// Warps per CTA and shared memory for their copy rings, per instantiation.
// More warps hide the per-block dependency chain; each warp keeps at least
// two stages so that one copy is in flight while it computes.  (Build-time
// overrides PKV_DECODE_WARPS / PKV_RING_KIB exist for tuning sweeps.)
template <int D, int G, int KV>
struct Tune {
#if defined(PKV_DECODE_WARPS) && defined(PKV_RING_KIB)
    static constexpr int NW = PKV_DECODE_WARPS;
    static constexpr int RING_KIB = PKV_RING_KIB;
#else
    // 4 warps, 48 KiB of stages: bf16 d128 keeps 2 stages of 8 KiB per warp
    // (3 CTAs = 12 warps per SM), FP8 d128 3 stages of 4 KiB (4 CTAs per SM).
    // Swept on GB300 over 2..8 warps and 32..128 KiB.
    static constexpr int NW = 4;
    // 4-bit: 36 KiB, 4 stages of 2176 bytes per warp at d_head 128 (two block
    // pairs), 8 of 1152 at d_head 64; its three CTAs per SM are held by
    // registers, not by shared memory.  Measured on GB300: 4 stages 61.6 us
    // per launch against 62.8 us with 8 (Llama3-8B shape, batch 128).
    static constexpr int RING_KIB = KV == 2 ? 36 : 48;
#endif
};

#ifndef PKV_I4_WARPS_PER_SM
#define PKV_I4_WARPS_PER_SM 12
#endif
#ifndef PKV_F8_WARPS_PER_SM
#define PKV_F8_WARPS_PER_SM 12
#endif

template <int D, int G, int KV>
struct Cfg {
    using Gm = Geo<D, KV>;
    static constexpr int NW = Tune<D, G, KV>::NW;
    static constexpr int kThreads = NW * 32;
    // resident CTAs per SM the register budget is held to: 12 warps per SM,
    // i.e. 3 x 128 threads of at most 168 registers for 4-warp CTAs (the
    // shared-memory ring allows no more for bf16 d128)
    static constexpr int kWarpsPerSm = KV == 2 ? PKV_I4_WARPS_PER_SM : KV == 1 ? PKV_F8_WARPS_PER_SM : 12;
    static constexpr int kMinBlocks = kWarpsPerSm / NW > 0 ? kWarpsPerSm / NW : 1;
    static constexpr int kStages = std::min(8, std::max(2, Tune<D, G, KV>::RING_KIB * 1024 / (NW * Gm::STAGE)));
    // shared-memory layout (bytes from a 1024-byte aligned base)
    static constexpr int kRing = NW * kStages * Gm::STAGE;
    static constexpr int kBars = kRing;
    static constexpr int kPhys = kBars + NW * kStages * 8;
    static constexpr int kNewRow = (kPhys + NW * kStages * 4 + 15) / 16 * 16;  // [NW][2 * D * 2] bytes:
                                                                                 // fused step's new rows
    static constexpr int kWarpTot = kNewRow + NW * 4 * D;
    // ps[batch + 1], then clamped lengths cl[batch], then table row starts rb[batch]
    static constexpr int kPs = kWarpTot + 4 * NW;
    static size_t smem_bytes(int batch) { return 1024 + (size_t)kPs + 4 * (size_t)(3 * batch + 1); }
    static_assert(G <= 8, "at most 8 query heads per KV head");
};

// Exclusive prefix sum of block counts per sequence (after the first `skip`
// table entries) into ps[0..batch], the clamped lengths into cl and each
// sequence's first table entry into rb (each if not null); range errors go
// to *err when err is not null.  A sequence's table row is W entries from
// b * W (dense form) or entries indptr[b] .. indptr[b+1] of n_indices (CSR
// form; a row outside that range counts as empty).  warp_tot is scratch for
// NW ints.  The decode and merge kernels both derive their work from it.
template <int NW>
__device__ void scan_blocks(const int32_t *lens, int batch, int W, const int32_t *indptr, int64_t n_indices,
                            int skip, unsigned *err, int32_t *ps, int32_t *cl, int32_t *rb, int *warp_tot)
{
    constexpr int NT = NW * 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int carry = 0;
    for (int base = 0; base < batch; base += NT) {
        const int b = base + tid;
        int n = 0;
        if (b < batch) {
            int c = lens[b];
            int width = W, row = b * W;
            if (indptr) {
                const int32_t lo = indptr[b], hi = indptr[b + 1];
                const bool ok = lo >= 0 && lo <= hi && (int64_t)hi <= n_indices;
                if (!ok && err) atomicOr(err, PKV_DEVERR_BLOCK_RANGE);
                width = ok ? hi - lo : 0;
                row = ok ? lo : 0;
            }
            if (rb) rb[b] = row;
            const int cmax = width > (INT32_MAX / kBlockSize) ? INT32_MAX : width * kBlockSize;
            if (c < 0 || c > cmax) {
                if (err) atomicOr(err, PKV_DEVERR_CTX_RANGE);
                c = c < 0 ? 0 : cmax;
            }
            if (c < skip * kBlockSize) {  // cascade: every sequence holds the whole prefix
                if (err) atomicOr(err, PKV_DEVERR_CTX_RANGE);
                c = skip * kBlockSize;
            }
            if (cl) cl[b] = c;
            n = (c + kBlockSize - 1) / kBlockSize - skip;  // blocks after the shared prefix
        }
        int x = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        int before = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int t = warp_tot[w];
            before += (w < warp) ? t : 0;
            tot += t;
        }
        if (b < batch) ps[b] = carry + before + x - n;
        carry += tot;
        __syncthreads();
    }
    if (tid == 0) ps[batch] = carry;
    __syncthreads();
}

// The stream: item f (0 <= f < total = n_kv * ps[batch]) is block j of head g
// of sequence b with f = n_kv * ps[b] + g * nblk_b + j.  Slice s covers items
// [s * share, (s + 1) * share); warp `me` of the grid takes slices me,
// me + n_warps, ...
struct Stream {
    const int32_t *ps;
    int batch, n_kv, total, share, n_slices, n_warps;
};

// One piece: blocks [j0, j1) of (b, g), starting at stream item f, in slice.
struct Piece {
    int b, g, j0, j1, nblk, f, slice;
};

__device__ __forceinline__ Piece locate(const Stream &st, int f, int slice)
{
    Piece p;
    int lo = 0, hi = st.batch - 1;  // largest b with n_kv * ps[b] <= f
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (st.n_kv * st.ps[mid] <= f) lo = mid; else hi = mid - 1;
    }
    p.b = lo;
    p.nblk = st.ps[lo + 1] - st.ps[lo];
    const int r = f - st.n_kv * st.ps[lo];
    p.g = r / p.nblk;
    p.j0 = r - p.g * p.nblk;
    const int slice_end = min(st.total, (slice + 1) * st.share);
    p.j1 = min(p.nblk, p.j0 + (slice_end - f));
    p.f = f;
    p.slice = slice;
    return p;
}

// The piece after p in this warp's walk.
__device__ __forceinline__ bool next_piece(const Stream &st, Piece &p)
{
    int f = p.f + (p.j1 - p.j0);
    int slice = p.slice;
    if (f >= min(st.total, (slice + 1) * st.share)) {
        slice += st.n_warps;
        if (slice >= st.n_slices) return false;
        f = slice * st.share;
    }
    p = locate(st, f, slice);
    return true;
}

__device__ __forceinline__ bool first_piece(const Stream &st, int me, Piece &p)
{
    if (me >= st.n_slices) return false;
    p = locate(st, me * st.share, me);
    return true;
}

// The producer walks the warp's blocks in segments of at most 32 consecutive
// blocks j .. j+n-1 of one piece.  One coalesced load fetches a segment's
// block-table entries (lane k holds block j+k's), one segment ahead of use,
// so no table read sits in front of a copy.
struct Seg {
    Piece p;
    int j, n;
    bool live;
};

__device__ __forceinline__ void seg_first(Seg &s, const Stream &st, int me)
{
    s.live = first_piece(st, me, s.p);
    s.j = s.live ? s.p.j0 : 0;
    s.n = s.live ? min(32, s.p.j1 - s.j) : 0;
}

__device__ __forceinline__ void seg_next(Seg &s, const Stream &st)
{
    if (!s.live) return;
    s.j += s.n;
    if (s.j >= s.p.j1) {
        s.live = next_piece(st, s.p);
        if (!s.live) {
            s.n = 0;
            return;
        }
        s.j = s.p.j0;
    }
    s.n = min(32, s.p.j1 - s.j);
}

__device__ __forceinline__ int seg_load(const Seg &s, int lane, const DecodeArgs &a, const int32_t *rb)
{
    return (s.live && lane < s.n) ? a.block_tables[(int64_t)rb[s.p.b] + a.skip_blocks + s.j + lane] : -1;
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core helpers (16x8x16 MMA, bf16 or f16 in, fp32 out)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    if constexpr (F16)
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
                     "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                     "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Slack (log2 units) of the decode softmax's lazy reference maximum: P <= 2^slack.
// 4-bit pools feed the MMA P times each token's value scale in f16, so their P
// stays small enough for f16 whatever the value range.
template <int KV>
constexpr float kRefSlack = KV == 2 ? 2.0f : 8.0f;

// 2^x with the MUFU approximation (relative error about 2^-22; results below
// 2^-126 flush to 0, 2^-inf = 0 and 2^0 = 1).  The decode softmax's weights use it.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Transpose an 8x8 matrix of 16-bit values held one row-pair per thread.
__device__ __forceinline__ uint32_t movm_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Four E4M3 bytes -> two f16x2 words (bytes 0,1 -> lo; bytes 2,3 -> hi); exact.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t &lo, uint32_t &hi)
{
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (F16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

// Byte offset inside a TMA box region (aligned to its swizzle atom) after the
// box's swizzle: 16-byte chunk index XOR the 128-byte line index (mod 8) for
// 128-byte rows, XOR (line index mod 4) for 64-byte rows.
template <int BOXB>
__device__ __forceinline__ uint32_t swz(uint32_t off)
{
    if constexpr (BOXB == 128) return off ^ ((off >> 3) & 0x70u);
    else if constexpr (BOXB == 64) return off ^ ((off >> 3) & 0x30u);
    else return off ^ ((off >> 3) & 0x10u);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Byte offset of (row, byte) offset `off` inside a stage's K or V tile: TMA
// boxes are swizzled, a 4-bit entry's bulk copy is not.
template <class Gm>
__device__ __forceinline__ uint32_t tile_off(uint32_t off)
{
    if constexpr (Gm::I4) return off;
    else return swz<Gm::BOXB>(off);
}

// 4-bit codes as f16 operands without a subtraction: a code c or-ed into
// the mantissa of 1024.0 is exactly 1024 + c (low nibble of each half word),
// or 1024 + 16 c (high nibble).  The decode kernel removes the offset and
// the factor where they do not cancel by themselves (see load_q_frags and
// the piece end).  The or-ed exponent bits come from constant memory, which
// the three-input logic instruction takes as an operand beside the mask
// immediate; written as a second immediate, the compiler put the constant
// into a register before each use, one more instruction per code pair (the
// 4-bit decode then issued a sixth more instructions and ran 14% slower).
__constant__ uint32_t kF16Exp1024 = 0x64006400u;  // 1024.0 in both halves of an f16 pair
__device__ __forceinline__ uint32_t i4_lo(uint32_t w) { return (w & 0x000F000Fu) | kF16Exp1024; }
__device__ __forceinline__ uint32_t i4_hi(uint32_t w) { return (w & 0x00F000F0u) | kF16Exp1024; }

// Byte `bi` of the packed words of two token rows a, b in half words 0 and 1
// of the result (row a low): i4_lo / i4_hi of it give the byte's two codes
// for both rows.
template <int bi>
__device__ __forceinline__ uint32_t i4_rows(uint32_t wa, uint32_t wb)
{
    constexpr uint32_t sel = bi | (bi << 4) | ((4 + bi) << 8) | ((4 + bi) << 12);
    return prmt(wa, wb, sel);
}

// q rows of one (sequence, KV head) group as m16n8k16 B fragments: thread
// (g8, c4) holds head g8's pairs of d for every k-step (zero for padding
// heads g8 >= G).  bf16 KV: k-step ks covers d 16ks + {2c, 2c+1} and
// 16ks + 8 + {2c, 2c+1}.  FP8 KV (f16 MMA): k-step 2kk+j covers
// d 32kk + 8c + 4j + {0,1} and {2,3}, the order the E4M3 K fragments use;
// they are left as loaded (bf16) for q_frags_to_f16.
// 4-bit KV (f16 MMA): q' = q * k_scale[g] per channel (the keys' per-channel
// scale folded into q; their zero points add the same constant to every
// score of a head and cancel in the softmax); k-step ks of thread c4 covers
// the channels of its packed key word w = ks / 2, base = c4 * D / 4 + 8w:
// pairs (base + s, base + s + 4), taken from the low nibbles of the word's
// half words (shifted right by 4s), and (base + s + 1, base + s + 5), from
// the high nibbles, with s = 2 * (ks & 1).  The keys enter the MMA as
// 1024 + c (low) and 1024 + 16 c (high), so the high channels' q' carries an
// exact factor 1/16; the offsets add sum_d 1024 q'_d, again one constant per
// head, which cancels in the softmax.
template <int D, int G, int KV>
__device__ __forceinline__ void load_q_frags(const DecodeArgs &a, int b, int g, int g8, int c4,
                                             uint32_t (&qf)[D / 16][2])
{
    constexpr bool FP8 = KV == kKvFp8, I4 = KV == kKvInt4;
    const bool live = g8 < G;
    const __nv_bfloat16 *qrow = a.q + ((int64_t)b * a.n_q + g * G + (live ? g8 : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        if constexpr (I4) {
            const int base = c4 * (D / 4) + 8 * (ks >> 1), s0 = 2 * (ks & 1);
            const float *sk = a.k_params + (int64_t)g * D + base + s0;
            const __nv_bfloat16 *qq = qrow + base + s0;
            // q' = q * k_scale * (scale * log2 e): the score scale folded in once per piece
            auto qv = [&](int k) { return live ? __bfloat162float(qq[k]) * sk[k] * a.qscale : 0.0f; };
            qf[ks][0] = pack2<true>(qv(0), qv(4));
            qf[ks][1] = pack2<true>(qv(1) * 0.0625f, qv(5) * 0.0625f);
        } else if constexpr (!FP8) {
            qf[ks][0] = live ? *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * c4) : 0u;
            qf[ks][1] = live ? *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 8 + 2 * c4) : 0u;
        } else {  // raw bf16 pairs; q_frags_to_f16 converts them when the piece starts
            const int d0 = 32 * (ks >> 1) + 8 * c4 + 4 * (ks & 1);
            const uint2 r = live ? *reinterpret_cast<const uint2 *>(qrow + d0) : make_uint2(0, 0);
            qf[ks][0] = r.x;
            qf[ks][1] = r.y;
        }
    }
}

// FP8 KV: the loaded bf16 pairs of q -> the f16 pairs the MMAs take (exact
// for |q| < 65504 apart from f16's shorter exponent range), done when the
// piece starts so that the load's latency stays hidden behind the piece
// before.
template <int D>
__device__ __forceinline__ void q_frags_to_f16(uint32_t (&qf)[D / 16][2])
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float2 x = bf16x2_to_f32x2(qf[ks][i]);
            qf[ks][i] = pack2<true>(x.x, x.y);
        }
}

// ---------------------------------------------------------------------------
// Merge of split runs: the split-KV reduction
//
// A (sequence, KV head) run that the decode kernel cut into several pieces
// (and, in cascade decode, every run) leaves partials (m, l, O) in workspace
// slots; this kernel, launched right behind the decode kernel, combines them
// by log-sum-exp in a fixed order (the n_pre prefix chunks, then the tail
// pieces in slice order):
//   M = max m_p,  L = sum 2^(m_p - M) l_p,  out = sum 2^(m_p - M) O_p / L.
// A run is split when its first and last blocks fall in different slices of
// the decode kernel's stream, which the kernel rederives from the lengths.
// One wave of CTAs walks the runs: two CTAs per run when the wave holds twice
// as many CTAs as runs (each warp summing an eighth of the run's G x D output
// columns), a CTA per run when it holds as many (a quarter each), else a
// warp per run.
// ---------------------------------------------------------------------------

constexpr int kMergeThreads = 128;
constexpr int kMergeWarps = kMergeThreads / 32;

struct MergeArgs {
    const float2 *ws_ml;
    const float *ws_o;
    __nv_bfloat16 *out;
    const int32_t *context_lens;
    const int32_t *indptr;  // CSR tables (null: dense)
    int64_t n_indices;
    int n_kv, n_q, batch, W, skip_blocks;
    int n_warps, slice_blocks;  // the decode grid's warps and slice length (0: automatic)
    int64_t pre_base;  // cascade: slot of prefix chunk 0 for (b=0, g=0); chunk k of (b, g) is
    int n_pre;         // pre_base + (k * batch + b) * n_kv + g; n_pre = 0 without a shared prefix
};

// One warp: chunks [c_lo, c_hi) (float4 chunks of the G x D output rows, at
// most CW of them) of run (b, g) with `np` pieces (n_pre prefix chunks, then
// tail slots from `base`).  Lane p reads piece p's (m, l) and keeps its
// weights, which lanes take by shuffle; PB pieces' rows are in flight at a
// time, the first PB requested together with the (m, l).  Every sum has a
// fixed order.
template <int D, int G, int CW>
__device__ __forceinline__ void merge_run_warp(const MergeArgs &a, int b, int g, int np, int64_t base, int c_lo,
                                               int c_hi, int lane)
{
    constexpr int KW = (CW + 31) / 32;  // chunks per lane
    constexpr int PB = 8 / KW;
    auto slot = [&](int p) -> int64_t {
        return p < a.n_pre ? a.pre_base + ((int64_t)p * a.batch + b) * a.n_kv + g : base + (p - a.n_pre);
    };
    auto load_o = [&](int p, float4 (&x)[KW]) {
        const float4 *src = reinterpret_cast<const float4 *>(a.ws_o + slot(p) * G * D);
#pragma unroll
        for (int k = 0; k < KW; ++k) {
            const int c = c_lo + lane + 32 * k;
            x[k] = c < c_hi ? __ldcg(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    float4 buf[PB][KW];
#pragma unroll
    for (int i = 0; i < PB; ++i)
        if (i < np) load_o(i, buf[i]);
    float own_m[G], lm[G], ll[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        own_m[h] = -INFINITY;
        lm[h] = -INFINITY;
        ll[h] = 0.0f;
    }
    for (int p0 = 0; p0 < np; p0 += 32) {
        if (p0 + lane < np) {
            const float2 *src = a.ws_ml + slot(p0 + lane) * G;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float2 v = __ldcg(src + h);
                if (p0 == 0) own_m[h] = v.x;
                const float mn = fmaxf(lm[h], v.x);
                ll[h] = mn == -INFINITY ? 0.0f : ll[h] * exp2f(lm[h] - mn) + v.y * exp2f(v.x - mn);
                lm[h] = mn;
            }
        }
    }
    float M[G], L[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float mx = lm[h];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
        float sl = mx == -INFINITY ? 0.0f : ll[h] * exp2f(lm[h] - mx);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) sl += __shfl_xor_sync(kFull, sl, off);
        M[h] = mx;
        L[h] = sl;
        own_m[h] = mx == -INFINITY ? 0.0f : exp2f(own_m[h] - mx);  // now the weight of piece `lane`
    }
    float4 acc[KW];
#pragma unroll
    for (int k = 0; k < KW; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < np; p += PB) {
#pragma unroll
        for (int i = 0; i < PB; ++i) {
            const int pi = p + i;
            if (pi < np) {
                float wv[G];
                if (pi < 32) {
#pragma unroll
                    for (int h = 0; h < G; ++h) wv[h] = __shfl_sync(kFull, own_m[h], pi);
                } else {
                    const float2 *src = a.ws_ml + slot(pi) * G;
#pragma unroll
                    for (int h = 0; h < G; ++h) wv[h] = M[h] == -INFINITY ? 0.0f : exp2f(__ldcg(src + h).x - M[h]);
                }
#pragma unroll
                for (int k = 0; k < KW; ++k) {
                    const int h = (c_lo + lane + 32 * k) * 4 / D;  // < G for chunks in range
                    float w = wv[0];
#pragma unroll
                    for (int hh = 1; hh < G; ++hh) w = h == hh ? wv[hh] : w;
                    acc[k].x = fmaf(w, buf[i][k].x, acc[k].x);
                    acc[k].y = fmaf(w, buf[i][k].y, acc[k].y);
                    acc[k].z = fmaf(w, buf[i][k].z, acc[k].z);
                    acc[k].w = fmaf(w, buf[i][k].w, acc[k].w);
                }
                if (pi + PB < np) load_o(pi + PB, buf[i]);
            }
        }
    }
    __nv_bfloat16 *ob = a.out + ((int64_t)b * a.n_q + g * G) * D;
#pragma unroll
    for (int k = 0; k < KW; ++k) {
        const int c = c_lo + lane + 32 * k;
        if (c < c_hi) {
            const int h = c * 4 / D;
            float Lh = L[0];
#pragma unroll
            for (int hh = 1; hh < G; ++hh) Lh = h == hh ? L[hh] : Lh;
            const float r = Lh > 0.0f ? 1.0f / Lh : 0.0f;
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x * r, acc[k].y * r);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z * r, acc[k].w * r);
            *reinterpret_cast<uint2 *>(ob + c * 4) =
                make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
        }
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kMergeThreads, 4) merge_kernel(MergeArgs a)
{
    constexpr int CHUNKS = G * D / 4;
    constexpr int CW = (CHUNKS + kMergeWarps - 1) / kMergeWarps;  // a CTA per run: columns per warp
    extern __shared__ int32_t ps[];  // [batch + 1]
    __shared__ int warp_tot[kMergeWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // The decode kernel's slicing, rederived from the lengths (its inputs, not
    // its outputs) while it still runs; only the partials need the wait.
    scan_blocks<kMergeWarps>(a.context_lens, a.batch, a.W, a.indptr, a.n_indices, a.skip_blocks, nullptr, ps,
                             nullptr, nullptr, warp_tot);
    const int total = a.n_kv * ps[a.batch];
    const int share = a.slice_blocks > 0 ? a.slice_blocks : max(1, (total + a.n_warps - 1) / a.n_warps);
    griddep_wait();  // the decode kernel's partials
    griddep_launch_dependents();
    const int runs = a.batch * a.n_kv;
    // (s_first, piece count) of run r; 0 pieces for an empty tail
    auto pieces = [&](int r, int &b, int &g, int &s_first) -> int {
        b = r / a.n_kv;
        g = r - b * a.n_kv;
        const int nblk = ps[b + 1] - ps[b];
        s_first = 0;
        if (nblk == 0) return 0;
        const int start = a.n_kv * ps[b] + g * nblk;
        s_first = start / share;
        return (start + nblk - 1) / share - s_first + 1;
    };
    if (2 * runs <= (int)gridDim.x) {  // two CTAs per run, each half of the columns: more pieces in flight
        constexpr int CW2 = (CHUNKS + 2 * kMergeWarps - 1) / (2 * kMergeWarps);
        const int r = blockIdx.x >> 1, half = blockIdx.x & 1;
        if (r >= runs) return;
        int b, g, s_first;
        const int n = pieces(r, b, g, s_first);
        if (a.n_pre == 0 && n <= 1) return;  // written whole by the decode kernel (or empty)
        const int c_lo = min(CHUNKS, (half * kMergeWarps + warp) * CW2), c_hi = min(CHUNKS, c_lo + CW2);
        const int64_t base = (int64_t)s_first + (int64_t)b * a.n_kv + g;  // slot of tail piece 0
        if (c_lo < c_hi) merge_run_warp<D, G, CW2>(a, b, g, a.n_pre + n, base, c_lo, c_hi, lane);
    } else if (runs <= (int)gridDim.x) {  // a CTA per run
        const int r = blockIdx.x;
        if (r >= runs) return;
        int b, g, s_first;
        const int n = pieces(r, b, g, s_first);
        if (a.n_pre == 0 && n <= 1) return;  // written whole by the decode kernel (or empty)
        const int c_lo = min(CHUNKS, warp * CW), c_hi = min(CHUNKS, c_lo + CW);
        const int64_t base = (int64_t)s_first + (int64_t)b * a.n_kv + g;  // slot of tail piece 0
        if (c_lo < c_hi) merge_run_warp<D, G, CW>(a, b, g, a.n_pre + n, base, c_lo, c_hi, lane);
    } else {  // a warp per run
        for (int r = blockIdx.x * kMergeWarps + warp; r < runs; r += gridDim.x * kMergeWarps) {
            int b, g, s_first;
            const int n = pieces(r, b, g, s_first);
            if (a.n_pre == 0 && n <= 1) continue;
            const int64_t base = (int64_t)s_first + (int64_t)b * a.n_kv + g;
            merge_run_warp<D, G, CHUNKS>(a, b, g, a.n_pre + n, base, 0, CHUNKS, lane);
        }
    }
}

// Fused step, part 1 (start of the piece that holds a sequence's last
// block): lane l < 2*NCH starts an asynchronous 16-byte copy of chunk l % NCH
// of the new K row (l < NCH) or V row into the warp's row buffer in shared
// memory, so nothing stays live in registers across the block loop.
template <int D>
__device__ __forceinline__ void fetch_new_row(const DecodeArgs &a, int b, int g, int lane, uint8_t *rowbuf)
{
    constexpr int NCH = D / 8;
    if (lane < 2 * NCH) {
        const __nv_bfloat16 *src = (lane >= NCH ? a.v_new : a.k_new) + ((int64_t)b * a.n_kv + g) * D + (lane % NCH) * 8;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(rowbuf + lane * 16)), "l"(src)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// ... and its bytes as the pool stores them: the bf16 copy, or for an E4M3
// pool E4M3(fp32(x) / scale) rounded to nearest even and saturated, from
// __fdiv_rn and a satfinite convert, exactly what paged_kv_append writes.
template <int D, int KV>
__device__ __forceinline__ uint4 prepared_new_row(const DecodeArgs &a, int g, int lane, const uint8_t *rowbuf)
{
    constexpr bool FP8 = KV == kKvFp8;
    constexpr int NCH = D / 8;
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    if (lane >= 2 * NCH) return make_uint4(0, 0, 0, 0);
    const uint4 chunk = *reinterpret_cast<const uint4 *>(rowbuf + lane * 16);
    if constexpr (!FP8) {
        return chunk;
    } else {
        const float sc = a.scales[(lane >= NCH ? a.n_kv : 0) + g];
        const uint32_t w[4] = {chunk.x, chunk.y, chunk.z, chunk.w};
        uint32_t q[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_f32x2(w[i]);
            const uint32_t e = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(f.x, sc), __fdiv_rn(f.y, sc)),
                                                        __NV_SATFINITE, __NV_E4M3);
            if (i & 1) q[i >> 1] |= e << 16;
            else q[i >> 1] = e;
        }
        return make_uint4(q[0], q[1], 0, 0);
    }
}

// Fused step, part 2 (when the block has landed): write the prepared row into
// the pool -- the append -- and into row r of the block's staged tiles, which
// the TMA filled before the append.
template <int D, int KV>
__device__ __forceinline__ void append_row(const DecodeArgs &a, int g, int phys, int r, int lane, uint4 prepared,
                                           uint8_t *stage)
{
    using Gm = Geo<D, KV>;
    constexpr bool FP8 = KV == kKvFp8;
    constexpr int NCH = D / 8;  // 8-element chunks per row
    if (lane >= 2 * NCH) return;
    const bool isv = lane >= NCH;
    const int c = lane % NCH;
    // pool row: key row r of the (block, KV head) entry, or its value row 16 rows further
    const int64_t row = ((int64_t)phys * a.n_kv + g) * 2 * kBlockSize + (isv ? kBlockSize : 0) + r;
    uint8_t *tile = stage + (isv ? Gm::VOFF : 0);
    if constexpr (!FP8) {
        // chunk c is 16 bytes of the 256/128-byte row: column range c / 8, 16-byte unit c % 8
        const uint32_t off = (c >> 3) * Gm::CSTRIDE + swz<128>(r * 128 + (c & 7) * 16);
        *reinterpret_cast<uint4 *>(tile + off) = prepared;
        *reinterpret_cast<uint4 *>(a.k_pool + row * D * 2 + c * 16) = prepared;
    } else {
        const uint2 q = make_uint2(prepared.x, prepared.y);
        *reinterpret_cast<uint2 *>(tile + swz<Gm::BOXB>(r * Gm::ROWB + c * 8)) = q;
        *reinterpret_cast<uint2 *>(a.k_pool + row * D + c * 8) = q;
    }
}

// Decode kernel: per-warp TMA ring, tensor-core scores and P.V.
//
// Per 16-token block a warp computes S^T[16 tokens x 8 heads] = K . Q^T with
// m16n8k16 MMAs (the G <= 8 query heads of the group are the N dimension,
// padded with zero rows of q), runs the online softmax on the accumulator
// fragments (thread: tokens g, g+8; heads 2c, 2c+1), turns P^T into the
// B operand with movmatrix, and accumulates O^T[d x heads] += V^T . P^T.
// bf16 KV: fragments come from ldmatrix (.trans for V) on the swizzled tiles.
// FP8 KV: bytes are read with 32/64-bit shared loads and converted to f16
// pairs in registers; the MMA's k (and, for V, its m) order is a fixed
// permutation of d applied identically to both operands and undone when the
// output is written, so the products are unchanged.
template <int D, int G, int KV, bool APPEND = false>
__global__ void __launch_bounds__(Cfg<D, G, KV>::kThreads, Cfg<D, G, KV>::kMinBlocks)
    decode_kernel(const __grid_constant__ CUtensorMap tm_kv, DecodeArgs a)
{
    using C = Cfg<D, G, KV>;
    using Gm = typename C::Gm;
    constexpr bool FP8 = KV == kKvFp8, I4 = KV == kKvInt4;
    static_assert(!(I4 && APPEND), "the fused step is not built for 4-bit pools");
    static_assert(!I4 || C::kStages >= 2, "4-bit pools take two ring stages per softmax step");
    constexpr int S = C::kStages;
    constexpr int NW = C::NW;
    constexpr int NT = D / 16;  // 16-wide MMA tiles along d
    constexpr int kThreads = C::kThreads;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, c4 = lane & 3;  // MMA fragment coordinates
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *ring = smem + warp * S * Gm::STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBars) + warp * S;
    int *phys_st = reinterpret_cast<int *>(smem + C::kPhys) + warp * S;
    int *warp_tot = reinterpret_cast<int *>(smem + C::kWarpTot);
    int32_t *ps = reinterpret_cast<int32_t *>(smem + C::kPs);
    uint8_t *rowbuf = smem + C::kNewRow + warp * 4 * D;  // fused step: this warp's new K and V rows

    if (tid == 0) {
        if constexpr (!I4) prefetch_tensormap(&tm_kv);  // 4-bit pools are read by bulk copies
        for (int i = 0; i < NW * S; ++i) mbar_init(reinterpret_cast<uint64_t *>(smem + C::kBars) + i, 1);
        fence_mbarrier_init();
    }
    int32_t *cl = ps + a.batch + 1;
    int32_t *rb = cl + a.batch;
    griddep_wait();  // inputs may come from the previous kernel on the stream
    griddep_launch_dependents();
    {
        // the block tables and q into L2, one 128-byte line per thread of the grid, while the
        // lengths are scanned: the warps' first table and q reads then hit L2
        const int64_t line = ((int64_t)blockIdx.x * kThreads + tid) * 128;
        const int64_t tab_bytes = 4 * (a.indptr ? a.n_indices : (int64_t)a.batch * a.W);
        if (line < tab_bytes) prefetch_l2(reinterpret_cast<const uint8_t *>(a.block_tables) + line);
        if (line < (int64_t)a.batch * a.n_q * D * 2) prefetch_l2(reinterpret_cast<const uint8_t *>(a.q) + line);
    }
    scan_blocks<NW>(a.context_lens, a.batch, a.W, a.indptr, a.n_indices, a.skip_blocks,
                    blockIdx.x == 0 ? a.err : nullptr, ps, cl, rb, warp_tot);  // ends with __syncthreads
    Stream st;
    st.ps = ps;
    st.batch = a.batch;
    st.n_kv = a.n_kv;
    st.total = a.n_kv * ps[a.batch];
    st.n_warps = (int)gridDim.x * NW;
    st.share = a.slice_blocks > 0 ? a.slice_blocks : max(1, (st.total + st.n_warps - 1) / st.n_warps);
    st.n_slices = (st.total + st.share - 1) / st.share;
    const int me = (int)blockIdx.x * NW + warp;
    if (a.n_pre == 0) {  // empty sequences: zero rows (cascade: the merge kernel writes them)
        for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
            if (ps[b + 1] != ps[b]) continue;
            uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t)b * a.n_q * D);
            for (int i = tid; i < a.n_q * D / 8; i += kThreads) o[i] = make_uint4(0, 0, 0, 0);
        }
    }

    const uint64_t policy = l2_policy_evict_first();
    bool aborted = false;
    int drain_from = -1;

    // ---- producer (uniform across the warp; lane 0 issues the copies) ----
    Seg cur;
    seg_first(cur, st, me);
    int tab_cur = seg_load(cur, lane, a, rb);
    Seg nxt = cur;
    seg_next(nxt, st);
    int tab_nxt = seg_load(nxt, lane, a, rb);
    int seg_k = 0, n_issued = 0;
    auto issue_next = [&]() {
        if (!cur.live) return;
        const int phys = __shfl_sync(kFull, tab_cur, seg_k);
        const int sidx = n_issued % S;
        if (lane == 0) {
            const bool ok = phys >= 0 && phys < a.num_blocks;
            phys_st[sidx] = ok ? phys : -1;
            if (ok) {
                const int64_t unit = (int64_t)phys * a.n_kv + cur.p.g;  // (block, KV head)
                uint8_t *dst = ring + sidx * Gm::STAGE;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[sidx], Gm::STAGE);
                if constexpr (I4) {
                    // the whole entry (key codes, value codes, value parameters) in one copy: one
                    // request stream per block instead of three (measured: the three small copies
                    // alone held the 4-bit stream to 72% of the copy peak)
                    bulk_g2s(dst, a.i4_entries + unit * Gm::STAGE, Gm::STAGE, &bars[sidx], policy);
                } else {
                    // the entry's 16 key and 16 value rows, one 32-row box per column range
                    const int y = (int)(unit * 2 * kBlockSize);
#pragma unroll
                    for (int r = 0; r < Gm::NREG; ++r)
                        tma_load_2d(dst + r * Gm::CSTRIDE, &tm_kv, r * Gm::BOX_ELEMS, y, &bars[sidx], policy);
                }
            } else {
                atomicOr(a.err, PKV_DEVERR_BLOCK_RANGE);
                mbar_arrive(&bars[sidx]);
            }
        }
        ++n_issued;
        if (++seg_k == cur.n) {
            cur = nxt;
            tab_cur = tab_nxt;
            seg_k = 0;
            seg_next(nxt, st);
            tab_nxt = seg_load(nxt, lane, a, rb);
        }
    };
    for (int i = 0; i < S; ++i) issue_next();

    // ldmatrix lane roles: K (A operand, rows = tokens) and V (A = V^T via .trans)
    const int row_k = (lane & 7) + ((lane >> 3) & 1) * 8, half_k = lane >> 4;
    const int row_v = (lane & 7) + (lane >> 4) * 8, half_v = (lane >> 3) & 1;
    // 4-bit stages: the thread's byte offsets in the K tile (row g8) and the V tile (row 2c); its
    // other rows (g8 + 8; 2c + 1, 2c + 8, 2c + 9) sit at whole-row distances from these
    [[maybe_unused]] const uint32_t k_off = g8 * Gm::ROWB + 4 * (D / 32) * c4;
    [[maybe_unused]] const uint32_t v_off = Gm::TILE + 2 * c4 * Gm::ROWB + 4 * (D / 64) * g8;

    Piece pc;
    bool have = first_piece(st, me, pc);
    uint32_t qn[NT][2];
    if constexpr (!I4)
        if (have) load_q_frags<D, G, KV>(a, pc.b, pc.g, g8, c4, qn);
    int consumed = 0;
    while (have) {
        Piece nx = pc;
        const bool have_nx = next_piece(st, nx);
        // q of head g8 of the group as MMA B fragments (zero for padding heads);
        // the next piece's are fetched now so their latency overlaps this one.
        // 4-bit pools load them when the piece starts instead: their pieces are
        // long (a quarter of a bf16 block's bytes per block) and the registers
        // of a second set are worth more as occupancy.
        uint32_t qf[NT][2];
        if constexpr (I4) {
            load_q_frags<D, G, KV>(a, pc.b, pc.g, g8, c4, qf);
        } else {
#pragma unroll
            for (int ks = 0; ks < NT; ++ks) {
                qf[ks][0] = qn[ks][0];
                qf[ks][1] = qn[ks][1];
            }
            if constexpr (FP8) q_frags_to_f16<D>(qf);  // before qn is loaded again
            if (have_nx) load_q_frags<D, G, KV>(a, nx.b, nx.g, g8, c4, qn);
        }
        const float qs = a.qscale * (FP8 ? a.scales[pc.g] : 1.0f);
        const int C_len = cl[pc.b];
        // Fused step: the warp owning the block of position C_len-1 appends the
        // new token (prepared here, written when that block has landed).
        const bool has_new = APPEND && pc.j1 == pc.nblk && C_len > 0;
        if constexpr (APPEND) {
            if (has_new) fetch_new_row<D>(a, pc.b, pc.g, lane, rowbuf);
        }
        float o[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.0f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;  // heads 2c, 2c+1
        float z0 = 0.0f, z1 = 0.0f;    // 4-bit: sum of p * (value zero point), heads 2c, 2c+1
        float zs0 = 0.0f, zs1 = 0.0f;  // 4-bit: sum of the f16 (p * value scale) the MMA used
        // Lazy reference maximum.  m0, m1 are reference maxima of heads 2c, 2c+1 (the same in
        // every lane of a head): a block's weights are 2^(s - m), and only when some lane's
        // scores (this thread's maxima lm0, lm1) pass a reference by more than kRefSlack does
        // the warp take the heads' maxima across lanes (three shuffle rounds), raise the
        // references and rescale l and O by al.  So P <= 2^kRefSlack and most blocks skip the
        // reduction.  The result is the same ratio sum p v / sum p in exact arithmetic.
        auto ref_update = [&](float lm0, float lm1, float &al0, float &al1) {
            if constexpr (KV != kKvFp8)  // FP8 pools take the maxima every block (measured faster there)
                if (!__any_sync(kFull, lm0 > m0 + kRefSlack<KV> || lm1 > m1 + kRefSlack<KV>)) return;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                lm0 = fmaxf(lm0, __shfl_xor_sync(kFull, lm0, off));
                lm1 = fmaxf(lm1, __shfl_xor_sync(kFull, lm1, off));
            }
            const float mn0 = fmaxf(m0, lm0), mn1 = fmaxf(m1, lm1);
            al0 = ex2_approx(m0 - mn0);  // 0 while the reference is -inf
            al1 = ex2_approx(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(kFull, al0 != 1.0f || al1 != 1.0f)) {
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    o[t][0] *= al0;
                    o[t][1] *= al1;
                    o[t][2] *= al0;
                    o[t][3] *= al1;
                }
            }
        };

        // One block: wait for its stage, (fused step, last block only) patch in
        // the new token, then scores, softmax and P.V.  The patching variant is
        // a separate instantiation so the hot loop carries no per-block check.
        auto block = [&](int j, auto patch) {
            const int sidx = consumed % S;
            const uint32_t parity = (uint32_t)(consumed / S) & 1u;
            if (!aborted) {
                const bool ok = mbar_wait_bounded(&bars[sidx], parity);
                aborted = __any_sync(kFull, !ok);
                if (aborted) {
                    drain_from = consumed;
                    if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
                }
            }
            if (!aborted && phys_st[sidx] >= 0) {
                const uint32_t kb = smem_u32(ring + sidx * Gm::STAGE);
                const uint32_t vb = kb + (I4 ? Gm::TILE : Gm::VOFF);
                const int nv = min(kBlockSize, C_len - (a.skip_blocks + j) * kBlockSize);
                if constexpr (decltype(patch)::value) {
                    append_row<D, KV>(a, pc.g, phys_st[sidx], nv - 1, lane,
                                       prepared_new_row<D, KV>(a, pc.g, lane, rowbuf), ring + sidx * Gm::STAGE);
                    __syncwarp();
                }
                // ---- S^T = K . Q^T ----
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (I4) {
                    // this thread's packed key words: channels c4*D/4 .. +D/4 of tokens g8, g8+8
                    constexpr int WPT = D / 32;
                    uint32_t kx[WPT], ky[WPT];
                    if constexpr (WPT == 4) {
                        const uint4 x = lds128(kb + tile_off<Gm>(g8 * Gm::ROWB + 16 * c4));
                        const uint4 y = lds128(kb + tile_off<Gm>((g8 + 8) * Gm::ROWB + 16 * c4));
                        kx[0] = x.x; kx[1] = x.y; kx[2] = x.z; kx[3] = x.w;
                        ky[0] = y.x; ky[1] = y.y; ky[2] = y.z; ky[3] = y.w;
                    } else {
                        const uint2 x = lds64(kb + tile_off<Gm>(g8 * Gm::ROWB + 8 * c4));
                        const uint2 y = lds64(kb + tile_off<Gm>((g8 + 8) * Gm::ROWB + 8 * c4));
                        kx[0] = x.x; kx[1] = x.y;
                        ky[0] = y.x; ky[1] = y.y;
                    }
#pragma unroll
                    for (int ks = 0; ks < NT; ++ks) {
                        const int w = ks >> 1;
                        const uint32_t x = (ks & 1) ? kx[w] >> 8 : kx[w], y = (ks & 1) ? ky[w] >> 8 : ky[w];
                        const uint32_t fa[4] = {i4_lo(x), i4_lo(y), i4_hi(x), i4_hi(y)};
                        mma16816<true>((ks & 1) ? sb : sa, fa, qf[ks][0], qf[ks][1]);
                    }
                } else if constexpr (!FP8) {
#pragma unroll
                    for (int ks = 0; ks < NT; ++ks) {
                        const int chunk = 2 * ks + half_k;
                        const uint32_t off = (chunk >> 3) * Gm::CSTRIDE + swz<128>(row_k * 128 + (chunk & 7) * 16);
                        uint32_t fa[4];
                        ldsm_x4(kb + off, fa);
                        mma16816<false>((ks & 1) ? sb : sa, fa, qf[ks][0], qf[ks][1]);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk) {
                        const uint32_t d0 = 32 * kk + 8 * c4;
                        const uint2 x = lds64(kb + swz<Gm::BOXB>(g8 * Gm::ROWB + d0));
                        const uint2 y = lds64(kb + swz<Gm::BOXB>((g8 + 8) * Gm::ROWB + d0));
                        uint32_t f0[4], f1[4];
                        e4m3x4_to_f16x4(x.x, f0[0], f0[2]);
                        e4m3x4_to_f16x4(y.x, f0[1], f0[3]);
                        e4m3x4_to_f16x4(x.y, f1[0], f1[2]);
                        e4m3x4_to_f16x4(y.y, f1[1], f1[3]);
                        mma16816<true>(sa, f0, qf[2 * kk][0], qf[2 * kk][1]);
                        mma16816<true>(sb, f1, qf[2 * kk + 1][0], qf[2 * kk + 1][1]);
                    }
                }
                float s[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) s[i] = I4 ? sa[i] + sb[i] : (sa[i] + sb[i]) * qs;  // 4-bit: qs is in q'

                if (g8 >= nv) s[0] = s[1] = -INFINITY;
                if (g8 + 8 >= nv) s[2] = s[3] = -INFINITY;
                // ---- online softmax (token 0 of a block is always valid), lazy reference maximum ----
                float al0 = 1.0f, al1 = 1.0f;
                ref_update(fmaxf(s[0], s[2]), fmaxf(s[1], s[3]), al0, al1);
                const float p0 = ex2_approx(s[0] - m0), p1 = ex2_approx(s[1] - m1);
                const float p2 = ex2_approx(s[2] - m0), p3 = ex2_approx(s[3] - m1);
                l0 = fmaf(l0, al0, p0 + p2);
                l1 = fmaf(l1, al1, p1 + p3);
                uint32_t pb0, pb1;  // P^T rows: tokens 2c, 2c+1 (pb0), 2c+8, 2c+9 (pb1) of head g
                if constexpr (I4) {
                    // v = c * s + z per token: P V = (P * s) C + (P . z); masked tokens weigh 0
                    const float2 *vps = reinterpret_cast<const float2 *>(ring + sidx * Gm::STAGE + Gm::PARAMS);
                    const float2 vp0 = g8 < nv ? vps[g8] : make_float2(0.f, 0.f);
                    const float2 vp1 = g8 + 8 < nv ? vps[g8 + 8] : make_float2(0.f, 0.f);
                    z0 = fmaf(z0, al0, fmaf(p0, vp0.y, p2 * vp1.y));
                    z1 = fmaf(z1, al1, fmaf(p1, vp0.y, p3 * vp1.y));
                    const uint32_t h0 = pack2<true>(p0 * vp0.x, p1 * vp0.x), h1 = pack2<true>(p2 * vp1.x, p3 * vp1.x);
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&h0));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&h1));
                    zs0 = fmaf(zs0, al0, f0.x + f1.x);
                    zs1 = fmaf(zs1, al1, f0.y + f1.y);
                    pb0 = movm_t(h0);
                    pb1 = movm_t(h1);
                } else {
                    pb0 = movm_t(pack2<FP8>(p0, p1));
                    pb1 = movm_t(pack2<FP8>(p2, p3));
                }
                // masked tokens' V must not reach the MMA (0 * non-finite garbage); 4-bit codes are finite
                [[maybe_unused]] const uint32_t mk01 =
                    (2 * c4 < nv ? 0x0000ffffu : 0u) | (2 * c4 + 1 < nv ? 0xffff0000u : 0u);
                [[maybe_unused]] const uint32_t mk23 =
                    (2 * c4 + 8 < nv ? 0x0000ffffu : 0u) | (2 * c4 + 9 < nv ? 0xffff0000u : 0u);
                // ---- O^T += V^T . P^T ----
                if constexpr (I4) {
                    // channels g8*D/8 .. +D/8 of tokens 2c, 2c+1, 2c+8, 2c+9: tile t row g8 is the span's
                    // channel t, row g8+8 its channel NT + t (codes are finite: no masking needed)
                    constexpr int WPR = D / 64;  // words per token row per thread (2 or 1)
                    uint32_t r0[WPR], r1[WPR], r2[WPR], r3[WPR];
                    const int rows[4] = {2 * c4, 2 * c4 + 1, 2 * c4 + 8, 2 * c4 + 9};
                    uint32_t *rr[4] = {r0, r1, r2, r3};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if constexpr (WPR == 2) {
                            const uint2 v = lds64(vb + tile_off<Gm>(rows[q] * Gm::ROWB + 8 * g8));
                            rr[q][0] = v.x;
                            rr[q][1] = v.y;
                        } else {
                            rr[q][0] = lds32(vb + tile_off<Gm>(rows[q] * Gm::ROWB + 4 * g8));
                        }
                    }
                    // tile t: byte t of the thread's span, row g8 its low code (channel 2t of the span),
                    // row g8 + 8 its high code (channel 2t + 1), as 1024 + c and 1024 + 16 c
                    auto tile = [&](auto tc) {
                        constexpr int t = decltype(tc)::value;
                        const uint32_t z01 = i4_rows<t % 4>(r0[t / 4], r1[t / 4]);
                        const uint32_t z23 = i4_rows<t % 4>(r2[t / 4], r3[t / 4]);
                        const uint32_t fa[4] = {i4_lo(z01), i4_hi(z01), i4_lo(z23), i4_hi(z23)};
                        mma16816<true>(o[t], fa, pb0, pb1);
                    };
                    tile(std::integral_constant<int, 0>{});
                    tile(std::integral_constant<int, 1>{});
                    tile(std::integral_constant<int, 2>{});
                    tile(std::integral_constant<int, 3>{});
                    if constexpr (NT == 8) {
                        tile(std::integral_constant<int, 4>{});
                        tile(std::integral_constant<int, 5>{});
                        tile(std::integral_constant<int, 6>{});
                        tile(std::integral_constant<int, 7>{});
                    }
                } else if constexpr (!FP8) {
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const int chunk = 2 * t + half_v;
                        const uint32_t off = (chunk >> 3) * Gm::CSTRIDE + swz<128>(row_v * 128 + (chunk & 7) * 16);
                        uint32_t fa[4];
                        ldsm_x4_t(vb + off, fa);
                        if (nv < kBlockSize) {
                            fa[0] &= mk01;
                            fa[1] &= mk01;
                            fa[2] &= mk23;
                            fa[3] &= mk23;
                        }
                        mma16816<false>(o[t], fa, pb0, pb1);
                    }
                } else {
                    // 8 bytes (d = 64 Q + 8 g8 .. + 7) of each of the thread's four token rows per load;
                    // each 4-byte half j feeds tiles 4 Q + 2 j (d + 4 j + {0, 1}) and 4 Q + 2 j + 1 (+ {2, 3})
#pragma unroll
                    for (int Q = 0; Q < D / 64; ++Q) {
                        const uint32_t db = 64 * Q + 8 * g8;
                        const uint2 v0 = lds64(vb + swz<Gm::BOXB>((2 * c4) * Gm::ROWB + db));
                        const uint2 v1 = lds64(vb + swz<Gm::BOXB>((2 * c4 + 1) * Gm::ROWB + db));
                        const uint2 v2 = lds64(vb + swz<Gm::BOXB>((2 * c4 + 8) * Gm::ROWB + db));
                        const uint2 v3 = lds64(vb + swz<Gm::BOXB>((2 * c4 + 9) * Gm::ROWB + db));
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint32_t r0 = j ? v0.y : v0.x, r1 = j ? v1.y : v1.x;
                            const uint32_t r2 = j ? v2.y : v2.x, r3 = j ? v3.y : v3.x;
                            uint32_t fa[4], fb[4];
                            e4m3x4_to_f16x4(prmt(r0, r1, 0x5140u), fa[0], fa[1]);  // d0, d1 of tokens 2c,2c+1
                            e4m3x4_to_f16x4(prmt(r0, r1, 0x7362u), fb[0], fb[1]);  // d2, d3
                            e4m3x4_to_f16x4(prmt(r2, r3, 0x5140u), fa[2], fa[3]);  // tokens 2c+8, 2c+9
                            e4m3x4_to_f16x4(prmt(r2, r3, 0x7362u), fb[2], fb[3]);
                            if (nv < kBlockSize) {
                                fa[0] &= mk01; fa[1] &= mk01; fa[2] &= mk23; fa[3] &= mk23;
                                fb[0] &= mk01; fb[1] &= mk01; fb[2] &= mk23; fb[3] &= mk23;
                            }
                            mma16816<true>(o[4 * Q + 2 * j], fa, pb0, pb1);
                            mma16816<true>(o[4 * Q + 2 * j + 1], fb, pb0, pb1);
                        }
                    }
                }
            }
            __syncwarp();
            ++consumed;
            if (!aborted) issue_next();
        };
        // 4-bit pools: two blocks per softmax step.  The 4-bit path is bound by each
        // warp's per-block chain, not by HBM (a block carries a quarter of a bf16 block's
        // bytes): one max, rescale decision and shuffle reduction for 32 tokens, and four
        // independent score MMA chains, per two stages.
        auto block2 = [&](int j) {
            const int s0i = consumed % S, s1i = (consumed + 1) % S;
            if (!aborted) {
                bool ok = mbar_wait_bounded(&bars[s0i], (uint32_t)(consumed / S) & 1u);
                ok = mbar_wait_bounded(&bars[s1i], (uint32_t)((consumed + 1) / S) & 1u) && ok;
                aborted = __any_sync(kFull, !ok);
                if (aborted) {
                    drain_from = consumed;
                    if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
                }
            }
            const bool ok0 = phys_st[s0i] >= 0, ok1 = phys_st[s1i] >= 0;
            if (!aborted && (ok0 || ok1)) {
                const uint32_t kb0 = smem_u32(ring + s0i * Gm::STAGE), kb1 = smem_u32(ring + s1i * Gm::STAGE);
                // valid tokens of each block (none for a block whose id was out of range)
                const int nv0 = ok0 ? min(kBlockSize, C_len - (a.skip_blocks + j) * kBlockSize) : 0;
                const int nv1 = ok1 ? min(kBlockSize, C_len - (a.skip_blocks + j + 1) * kBlockSize) : 0;
                constexpr int WPT = D / 32;  // packed key words per token row per thread
                float sa0[4] = {0.f, 0.f, 0.f, 0.f}, sb0[4] = {0.f, 0.f, 0.f, 0.f};
                float sa1[4] = {0.f, 0.f, 0.f, 0.f}, sb1[4] = {0.f, 0.f, 0.f, 0.f};
                // the thread's packed key words two at a time (8 bytes of each of its two token rows
                // per block), so that only eight of them are live at once
                const uint32_t ka0 = kb0 + k_off, ka1 = kb1 + k_off;
#pragma unroll
                for (int hh = 0; hh < WPT / 2; ++hh) {
                    // rows g8 and g8 + 8 of each block, 8 bytes at a time
                    const uint2 kx0 = lds64(ka0 + 8 * hh), ky0 = lds64(ka0 + 8 * Gm::ROWB + 8 * hh);
                    const uint2 kx1 = lds64(ka1 + 8 * hh), ky1 = lds64(ka1 + 8 * Gm::ROWB + 8 * hh);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int ks = 4 * hh + k4;
                        const bool second = (k4 >> 1) != 0;  // word 2 hh + 1
                        const uint32_t wx0 = second ? kx0.y : kx0.x, wy0 = second ? ky0.y : ky0.x;
                        const uint32_t wx1 = second ? kx1.y : kx1.x, wy1 = second ? ky1.y : ky1.x;
                        const uint32_t x0 = (ks & 1) ? wx0 >> 8 : wx0, y0 = (ks & 1) ? wy0 >> 8 : wy0;
                        const uint32_t x1 = (ks & 1) ? wx1 >> 8 : wx1, y1 = (ks & 1) ? wy1 >> 8 : wy1;
                        const uint32_t fa0[4] = {i4_lo(x0), i4_lo(y0), i4_hi(x0), i4_hi(y0)};
                        const uint32_t fa1[4] = {i4_lo(x1), i4_lo(y1), i4_hi(x1), i4_hi(y1)};
                        mma16816<true>((ks & 1) ? sb0 : sa0, fa0, qf[ks][0], qf[ks][1]);
                        mma16816<true>((ks & 1) ? sb1 : sa1, fa1, qf[ks][0], qf[ks][1]);
                    }
                }
                // s[0..3]: block 0 (tokens g8, g8 + 8 x heads 2c, 2c+1), s[4..7]: block 1
                float s[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    s[i] = sa0[i] + sb0[i];  // the score scale is folded into q'
                    s[4 + i] = sa1[i] + sb1[i];
                }
                if (g8 >= nv0) s[0] = s[1] = -INFINITY;
                if (g8 + 8 >= nv0) s[2] = s[3] = -INFINITY;
                if (g8 >= nv1) s[4] = s[5] = -INFINITY;
                if (g8 + 8 >= nv1) s[6] = s[7] = -INFINITY;
                // ---- online softmax over the 32 tokens (a valid block has a valid token 0),
                // lazy reference maximum ----
                float al0 = 1.0f, al1 = 1.0f;
                ref_update(fmaxf(fmaxf(s[0], s[2]), fmaxf(s[4], s[6])), fmaxf(fmaxf(s[1], s[3]), fmaxf(s[5], s[7])),
                           al0, al1);
                float p[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) p[i] = ex2_approx(s[i] - ((i & 1) ? m1 : m0));
                l0 = fmaf(l0, al0, (p[0] + p[2]) + (p[4] + p[6]));
                l1 = fmaf(l1, al1, (p[1] + p[3]) + (p[5] + p[7]));
                // v = c * s + z per token: P V = (P * s) C + (P . z); masked tokens weigh 0
                const float2 zero2 = make_float2(0.f, 0.f);
                const float2 *vps0 = reinterpret_cast<const float2 *>(ring + s0i * Gm::STAGE + Gm::PARAMS);
                const float2 *vps1 = reinterpret_cast<const float2 *>(ring + s1i * Gm::STAGE + Gm::PARAMS);
                const float2 vp00 = g8 < nv0 ? vps0[g8] : zero2;
                const float2 vp01 = g8 + 8 < nv0 ? vps0[g8 + 8] : zero2;
                const float2 vp10 = g8 < nv1 ? vps1[g8] : zero2;
                const float2 vp11 = g8 + 8 < nv1 ? vps1[g8 + 8] : zero2;
                z0 = fmaf(z0, al0, fmaf(p[0], vp00.y, p[2] * vp01.y) + fmaf(p[4], vp10.y, p[6] * vp11.y));
                z1 = fmaf(z1, al1, fmaf(p[1], vp00.y, p[3] * vp01.y) + fmaf(p[5], vp10.y, p[7] * vp11.y));
                const uint32_t h00 = pack2<true>(p[0] * vp00.x, p[1] * vp00.x);
                const uint32_t h01 = pack2<true>(p[2] * vp01.x, p[3] * vp01.x);
                const uint32_t h10 = pack2<true>(p[4] * vp10.x, p[5] * vp10.x);
                const uint32_t h11 = pack2<true>(p[6] * vp11.x, p[7] * vp11.x);
                const float2 f00 = __half22float2(*reinterpret_cast<const __half2 *>(&h00));
                const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
                const float2 f10 = __half22float2(*reinterpret_cast<const __half2 *>(&h10));
                const float2 f11 = __half22float2(*reinterpret_cast<const __half2 *>(&h11));
                zs0 = fmaf(zs0, al0, (f00.x + f01.x) + (f10.x + f11.x));
                zs1 = fmaf(zs1, al1, (f00.y + f01.y) + (f10.y + f11.y));
                const uint32_t pb00 = movm_t(h00), pb01 = movm_t(h01), pb10 = movm_t(h10), pb11 = movm_t(h11);
                // ---- O^T += V^T . P^T, both blocks (codes are finite: no masking needed) ----
                constexpr int WPR = D / 64;  // words per token row per thread (2 or 1)
                // one packed value word of each of the thread's four token rows per block at a time
                // (tiles 4 w .. 4 w + 3 use word w), so that only eight words are live at once
                // rows 2c, 2c + 1, 2c + 8, 2c + 9: row distances 0, 1, 8, 9 from row 2c
                constexpr int kVRow[4] = {0, 1, 8, 9};
                auto vword = [&](uint32_t va, int q, int w) { return lds32(va + kVRow[q] * Gm::ROWB + 4 * w); };
                const uint32_t va0 = kb0 + v_off, va1 = kb1 + v_off;
                auto tile2 = [&](auto tc, const uint32_t (&u)[4], const uint32_t (&v)[4]) {
                    constexpr int t = decltype(tc)::value;
                    const uint32_t za = i4_rows<t % 4>(u[0], u[1]), zb = i4_rows<t % 4>(u[2], u[3]);
                    const uint32_t zc = i4_rows<t % 4>(v[0], v[1]), zd = i4_rows<t % 4>(v[2], v[3]);
                    const uint32_t fa[4] = {i4_lo(za), i4_hi(za), i4_lo(zb), i4_hi(zb)};
                    const uint32_t fb[4] = {i4_lo(zc), i4_hi(zc), i4_lo(zd), i4_hi(zd)};
                    mma16816<true>(o[t], fa, pb00, pb01);
                    mma16816<true>(o[t], fb, pb10, pb11);
                };
                {
                    const uint32_t u[4] = {vword(va0, 0, 0), vword(va0, 1, 0), vword(va0, 2, 0), vword(va0, 3, 0)};
                    const uint32_t v[4] = {vword(va1, 0, 0), vword(va1, 1, 0), vword(va1, 2, 0), vword(va1, 3, 0)};
                    tile2(std::integral_constant<int, 0>{}, u, v);
                    tile2(std::integral_constant<int, 1>{}, u, v);
                    tile2(std::integral_constant<int, 2>{}, u, v);
                    tile2(std::integral_constant<int, 3>{}, u, v);
                }
                if constexpr (NT == 8) {
                    const uint32_t u[4] = {vword(va0, 0, 1), vword(va0, 1, 1), vword(va0, 2, 1), vword(va0, 3, 1)};
                    const uint32_t v[4] = {vword(va1, 0, 1), vword(va1, 1, 1), vword(va1, 2, 1), vword(va1, 3, 1)};
                    tile2(std::integral_constant<int, 4>{}, u, v);
                    tile2(std::integral_constant<int, 5>{}, u, v);
                    tile2(std::integral_constant<int, 6>{}, u, v);
                    tile2(std::integral_constant<int, 7>{}, u, v);
                }
            }
            __syncwarp();
            consumed += 2;
            if (!aborted) {
                issue_next();
                issue_next();
            }
        };
        const int j_plain = has_new ? pc.j1 - 1 : pc.j1;  // has_new: the piece ends with the last block
        int j = pc.j0;
        if constexpr (I4) {
            for (; j + 1 < j_plain; j += 2) block2(j);
        }
        for (; j < j_plain; ++j) block(j, std::false_type{});
        if constexpr (APPEND) {
            if (has_new) block(j_plain, std::true_type{});
        }

        // ---- piece end ----
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, off);
            l1 += __shfl_xor_sync(kFull, l1, off);
        }
        if constexpr (I4) {
            // the MMA summed (P * s)(1024 + c) over low codes and (P * s)(1024 + 16 c) over high
            // ones: take off 1024 sum (P * s), undo the 16, and add the values' zero points'
            // sum_p p_p z_p (the same for every channel)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                z0 += __shfl_xor_sync(kFull, z0, off);
                z1 += __shfl_xor_sync(kFull, z1, off);
                zs0 += __shfl_xor_sync(kFull, zs0, off);
                zs1 += __shfl_xor_sync(kFull, zs1, off);
            }
            const float c0 = 1024.0f * zs0, c1 = 1024.0f * zs1;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                o[t][0] = (o[t][0] - c0) + z0;
                o[t][1] = (o[t][1] - c1) + z1;
                o[t][2] = (o[t][2] - c0) * 0.0625f + z0;
                o[t][3] = (o[t][3] - c1) * 0.0625f + z1;
            }
        }
        // channel of accumulator row g8 + 8i of tile t, per KV type
        auto chan = [&](int t, int i) {
            return I4 ? g8 * (D / 8) + 2 * t + i : FP8 ? 64 * (t >> 2) + 8 * g8 + 2 * (t & 3) + i : 16 * t + g8 + 8 * i;
        };
        const float vs = FP8 ? a.scales[a.n_kv + pc.g] : 1.0f;
        const bool h0 = 2 * c4 < G, h1 = 2 * c4 + 1 < G;  // this thread's heads exist
        if (pc.j0 == 0 && pc.j1 == pc.nblk && a.n_pre == 0) {
            // the whole (b, g): normalise and write bf16 out
            const float r0 = l0 > 0.0f ? vs / l0 : 0.0f, r1 = l1 > 0.0f ? vs / l1 : 0.0f;
            __nv_bfloat16 *ob = a.out + ((int64_t)pc.b * a.n_q + pc.g * G) * D;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int d = chan(t, i);
                    if (h0) ob[(2 * c4) * D + d] = __float2bfloat16_rn(o[t][2 * i] * r0);
                    if (h1) ob[(2 * c4 + 1) * D + d] = __float2bfloat16_rn(o[t][2 * i + 1] * r1);
                }
            }
        } else {
            // a part of (b, g) (or, in cascade decode, its tail): publish (m, l, O)
            // for the merge kernel
            const int64_t slot = (int64_t)pc.slice + (int64_t)pc.b * a.n_kv + pc.g;  // unique along the stream
            float *wo = a.ws_o + slot * G * D;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int d = chan(t, i);
                    if (h0) wo[(2 * c4) * D + d] = o[t][2 * i] * vs;
                    if (h1) wo[(2 * c4 + 1) * D + d] = o[t][2 * i + 1] * vs;
                }
            }
            if (g8 == 0) {
                if (h0) a.ws_ml[slot * G + 2 * c4] = make_float2(m0, l0);
                if (h1) a.ws_ml[slot * G + 2 * c4 + 1] = make_float2(m1, l1);
            }
        }
        pc = nx;
        have = have_nx;
    }

    if (drain_from >= 0)  // copies may still be in flight only after a timeout
        for (int k = drain_from; k < n_issued; ++k)
            mbar_wait_bounded(&bars[k % S], (uint32_t)(k / S) & 1u, 100000000ull);
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: partial (max, sum) and O for up to n_slices + batch * n_kv
// pieces.  Nothing in it needs to start at zero: every partial the merge
// kernel reads was written by the decode launch before it.
struct WsLayout {
    size_t ml, o, total;
};

static WsLayout ws_layout(int n_q, int n_kv, int d_head, int64_t slots)
{
    const int G = n_q / n_kv;
    WsLayout w;
    w.ml = 0;
    w.o = w.ml + align256(8 * (size_t)slots * G);
    w.total = w.o + 4 * (size_t)slots * G * d_head;
    return w;
}

// Upper bound on the slices of the stream; `warps` is the grid's total warp
// count.
static int64_t max_slices(pkv_pool *pool, int batch, int n_kv, int max_blocks_per_seq, int warps)
{
    const int slice_blocks = pool->partition_tokens / kBlockSize;
    const int64_t total = (int64_t)batch * n_kv * max_blocks_per_seq;
    return slice_blocks > 0 ? (total + slice_blocks - 1) / slice_blocks : (int64_t)warps;
}

// Upper bound on pieces (workspace slots): one per slice plus one per
// (sequence, head) run.
static int64_t max_slots(pkv_pool *pool, int batch, int n_kv, int max_blocks_per_seq, int warps)
{
    return max_slices(pool, batch, n_kv, max_blocks_per_seq, warps) + (int64_t)batch * n_kv;
}

// Persistent grid of the decode kernel for (d_head, G, dtype) at `batch`.
template <int D, int G, int KV, bool APPEND = false>
static pkv_status decode_grid(pkv_pool *pool, int batch, int max_blocks_per_seq, int *grid, size_t *smem)
{
    using C = Cfg<D, G, KV>;
    auto kern = decode_kernel<D, G, KV, APPEND>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        // The opt-in limit covers static plus dynamic shared memory.
        int optin = 0;
        cudaFuncAttributes fa;
        attr_err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, pool->device);
        if (attr_err == cudaSuccess) attr_err = cudaFuncGetAttributes(&fa, kern);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            optin - (int)fa.sharedSizeBytes);
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(decode)");
    *smem = C::smem_bytes(batch);
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::kThreads, *smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (occ < 1) return fail(PKV_EUNSUPPORTED, "decode: %zu bytes of shared memory do not fit", *smem);
    // At most every resident CTA, and no more CTAs than give each warp about
    // kMinBlocksPerWarp blocks of the largest possible batch, so that small
    // batches do not pay for launching and merging across idle warps.
    const int64_t ub_blocks = (int64_t)batch * pool->n_kv * max_blocks_per_seq;
    const int64_t want = (ub_blocks + (int64_t)C::NW * kMinBlocksPerWarp - 1) / ((int64_t)C::NW * kMinBlocksPerWarp);
    *grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)pool->num_sms * occ, want));
    return PKV_OK;
}

// Point the decode arguments at workspace `ws` laid out as L.
static void bind_workspace(DecodeArgs &a, uint8_t *ws, const WsLayout &L)
{
    a.ws_ml = reinterpret_cast<float2 *>(ws + L.ml);
    a.ws_o = reinterpret_cast<float *>(ws + L.o);
}

// The merge kernel behind a decode launch with arguments `a` on a grid of
// n_warps warps; its CTAs wait (programmatic dependent launch) for the
// decode grid to finish.
template <int D, int G>
static pkv_status launch_merge(pkv_pool *pool, const DecodeArgs &a, int n_warps, cudaStream_t s)
{
    MergeArgs m;
    m.ws_ml = a.ws_ml;
    m.ws_o = a.ws_o;
    m.out = a.out;
    m.context_lens = a.context_lens;
    m.n_kv = a.n_kv;
    m.n_q = a.n_q;
    m.batch = a.batch;
    m.W = a.W;
    m.indptr = a.indptr;
    m.n_indices = a.n_indices;
    m.skip_blocks = a.skip_blocks;
    m.n_warps = n_warps;
    m.slice_blocks = a.slice_blocks;
    m.pre_base = a.pre_base;
    m.n_pre = a.n_pre;
    static int occ = 0;
    static std::once_flag once;
    const size_t smem = 4 * ((size_t)a.batch + 1);
    std::call_once(once, [&] {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, merge_kernel<D, G>, kMergeThreads,
                                                          4 * (kMaxBatch + 1)) != cudaSuccess)
            occ = 1;
    });
    // one wave: as many CTAs as are resident at once; two per run while that fits, else at most one per run
    const int64_t runs = (int64_t)a.batch * a.n_kv;
    const int64_t slots = (int64_t)pool->num_sms * std::max(1, occ);
    const int grid = (int)std::max<int64_t>(1, 2 * runs <= slots ? 2 * runs : std::min<int64_t>(runs, slots));
    LaunchScope ls(pool, kMerge, s);
    cudaError_t e = launch_pdl(merge_kernel<D, G>, dim3((unsigned)grid), dim3(kMergeThreads), smem, s, m);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return PKV_OK;
}

template <int D, int G, int KV>
static pkv_status launch_decode(pkv_pool *pool, DecodeArgs a, cudaStream_t s)
{
    using C = Cfg<D, G, KV>;
    int grid = 0;
    size_t smem = 0;
    pkv_status st = decode_grid<D, G, KV>(pool, a.batch, a.W, &grid, &smem);
    if (st != PKV_OK) return st;
    const WsLayout L = ws_layout(a.n_q, a.n_kv, D, max_slots(pool, a.batch, a.n_kv, a.W, grid * C::NW));
    st = ensure_workspace(pool, L.total);
    if (st != PKV_OK) return st;
    bind_workspace(a, static_cast<uint8_t *>(pool->ws), L);
    LaunchScope ls(pool, kDecode, s);
    cudaError_t e = launch_pdl(decode_kernel<D, G, KV>, dim3(grid), dim3(C::kThreads), smem, s, pool->tm_entry,
                               a);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return launch_merge<D, G>(pool, a, grid * C::NW, s);
}

template <int D, int KV>
static pkv_status dispatch_g(pkv_pool *pool, const DecodeArgs &a, int G, cudaStream_t s);

// The decode launch for the pool's KV type and head size.
static pkv_status dispatch_kv(pkv_pool *pool, const DecodeArgs &a, int G, cudaStream_t s)
{
    const bool d128 = pool->d_head == 128;
    if (pool->dtype == PKV_INT4)
        return d128 ? dispatch_g<128, kKvInt4>(pool, a, G, s) : dispatch_g<64, kKvInt4>(pool, a, G, s);
    if (pool->dtype == PKV_FP8_E4M3)
        return d128 ? dispatch_g<128, kKvFp8>(pool, a, G, s) : dispatch_g<64, kKvFp8>(pool, a, G, s);
    return d128 ? dispatch_g<128, kKvBf16>(pool, a, G, s) : dispatch_g<64, kKvBf16>(pool, a, G, s);
}

template <int D, int KV>
static pkv_status dispatch_g(pkv_pool *pool, const DecodeArgs &a, int G, cudaStream_t s)
{
    switch (G) {
    case 1: return launch_decode<D, 1, KV>(pool, a, s);
    case 2: return launch_decode<D, 2, KV>(pool, a, s);
    case 4: return launch_decode<D, 4, KV>(pool, a, s);
    case 8: return launch_decode<D, 8, KV>(pool, a, s);
    }
    return fail(PKV_EUNSUPPORTED, "decode: group size %d unsupported (1, 2, 4 or 8)", G);
}

// Total warps of the decode grid (the larger of the plain and fused-step
// kernels, which may differ in occupancy).
template <int D, int G, int KV>
static pkv_status grid_warps(pkv_pool *pool, int batch, int max_blocks_per_seq, int *warps)
{
    size_t smem = 0;
    int g0 = 0, g1 = 0;
    pkv_status st = decode_grid<D, G, KV>(pool, batch, max_blocks_per_seq, &g0, &smem);
    if constexpr (KV != kKvInt4)  // the fused step's grid (no fused step for 4-bit pools)
        if (st == PKV_OK) st = decode_grid<D, G, KV, true>(pool, batch, max_blocks_per_seq, &g1, &smem);
    *warps = std::max(g0, g1) * Cfg<D, G, KV>::NW;
    return st;
}

template <int D, int KV>
static pkv_status grid_g(pkv_pool *pool, int G, int batch, int max_blocks_per_seq, int *warps)
{
    switch (G) {
    case 1: return grid_warps<D, 1, KV>(pool, batch, max_blocks_per_seq, warps);
    case 2: return grid_warps<D, 2, KV>(pool, batch, max_blocks_per_seq, warps);
    case 4: return grid_warps<D, 4, KV>(pool, batch, max_blocks_per_seq, warps);
    case 8: return grid_warps<D, 8, KV>(pool, batch, max_blocks_per_seq, warps);
    }
    return fail(PKV_EUNSUPPORTED, "decode: group size %d unsupported (1, 2, 4 or 8)", G);
}

// Workspace bytes a decode call with these sizes needs on this pool.
pkv_status decode_workspace_bytes(pkv_pool *pool, int batch, int n_q, int max_blocks_per_seq, size_t *bytes)
{
    const int G = n_q / pool->n_kv;
    int warps = 0;
    const int W = max_blocks_per_seq;
    const bool d128 = pool->d_head == 128;
    pkv_status st;
    if (pool->dtype == PKV_INT4)
        st = d128 ? grid_g<128, kKvInt4>(pool, G, batch, W, &warps) : grid_g<64, kKvInt4>(pool, G, batch, W, &warps);
    else if (pool->dtype == PKV_FP8_E4M3)
        st = d128 ? grid_g<128, kKvFp8>(pool, G, batch, W, &warps) : grid_g<64, kKvFp8>(pool, G, batch, W, &warps);
    else
        st = d128 ? grid_g<128, kKvBf16>(pool, G, batch, W, &warps) : grid_g<64, kKvBf16>(pool, G, batch, W, &warps);
    if (st != PKV_OK) return st;
    *bytes = ws_layout(n_q, pool->n_kv, pool->d_head,
                       max_slots(pool, batch, pool->n_kv, max_blocks_per_seq, warps)).total;
    return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_decode_attention(pkv_pool *pool, const void *q, int32_t n_q,
                                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                                             const int32_t *context_lens, int32_t batch, float scale,
                                             void *out, void *stream)
{
    if (!pool) return fail(PKV_EINVAL, "paged_decode_attention: NULL pool");
    if (batch < 0) return fail(PKV_EINVAL, "paged_decode_attention: batch < 0");
    if (n_q <= 0 || n_q % pool->n_kv)
        return fail(PKV_EINVAL, "paged_decode_attention: n_q %d is not a positive multiple of n_kv %d", n_q,
                    pool->n_kv);
    const int G = n_q / pool->n_kv;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention: n_q / n_kv = %d unsupported (1, 2, 4, 8)", G);
    if (max_blocks_per_seq <= 0 || max_blocks_per_seq > (1 << 24))
        return fail(PKV_EINVAL, "paged_decode_attention: max_blocks_per_seq %d out of range", max_blocks_per_seq);
    if (!isfinite(scale)) return fail(PKV_EINVAL, "paged_decode_attention: scale is not finite");
    if (batch == 0) return PKV_OK;
    if (batch > kMaxBatch)
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention: batch %d > %d", batch, kMaxBatch);
    if ((int64_t)batch * pool->n_kv * max_blocks_per_seq >= ((int64_t)1 << 30))
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention: batch x n_kv x max_blocks_per_seq too large");
    if (!q || !block_tables || !context_lens || !out)
        return fail(PKV_EINVAL, "paged_decode_attention: NULL device pointer");
    if (((uintptr_t)q | (uintptr_t)out) & 15u)
        return fail(PKV_EINVAL, "paged_decode_attention: q and out must be 16-byte aligned");
    if (((uintptr_t)block_tables | (uintptr_t)context_lens) & 3u)
        return fail(PKV_EINVAL, "paged_decode_attention: tables and lengths must be 4-byte aligned");
    if (!pool->scales_set && pool->dtype != PKV_BF16)
        return fail(PKV_EINVAL, "paged_decode_attention: %s pool needs its %s first",
                    pool->dtype == PKV_INT4 ? "4-bit" : "FP8",
                    pool->dtype == PKV_INT4 ? "kv_pool_set_int4_key_params" : "kv_pool_set_fp8_scales");

    DecodeArgs a;
    a.num_blocks = pool->num_blocks;
    a.n_kv = pool->n_kv;
    a.n_q = n_q;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.W = max_blocks_per_seq;
    a.indptr = nullptr;
    a.n_indices = 0;
    a.context_lens = context_lens;
    a.batch = batch;
    a.qscale = scale * kLog2e;
    a.scales = pool->scales;
    a.k_params = pool->k_params;
    a.i4_entries = pool->dtype == PKV_INT4 ? static_cast<const uint8_t *>(pool->k) : nullptr;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.ws_ml = nullptr;
    a.ws_o = nullptr;
    a.slice_blocks = pool->partition_tokens / kBlockSize;
    a.err = pool->err;
    a.k_new = a.v_new = nullptr;
    a.k_pool = nullptr;
    a.skip_blocks = 0;
    a.n_pre = 0;
    a.pre_base = 0;
    return dispatch_kv(pool, a, G, static_cast<cudaStream_t>(stream));
}

extern "C" pkv_status paged_decode_attention_csr(pkv_pool *pool, const void *q, int32_t n_q,
                                                 const int32_t *kv_indptr, const int32_t *kv_indices,
                                                 int64_t n_indices, const int32_t *context_lens, int32_t batch,
                                                 float scale, void *out, void *stream)
{
    if (!pool) return fail(PKV_EINVAL, "paged_decode_attention_csr: NULL pool");
    if (batch < 0) return fail(PKV_EINVAL, "paged_decode_attention_csr: batch < 0");
    if (n_q <= 0 || n_q % pool->n_kv)
        return fail(PKV_EINVAL, "paged_decode_attention_csr: n_q %d is not a positive multiple of n_kv %d", n_q,
                    pool->n_kv);
    const int G = n_q / pool->n_kv;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention_csr: n_q / n_kv = %d unsupported (1, 2, 4, 8)", G);
    if (n_indices < 0) return fail(PKV_EINVAL, "paged_decode_attention_csr: n_indices < 0");
    if (!isfinite(scale)) return fail(PKV_EINVAL, "paged_decode_attention_csr: scale is not finite");
    if (batch == 0) return PKV_OK;
    if (batch > kMaxBatch)
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention_csr: batch %d > %d", batch, kMaxBatch);
    if ((int64_t)pool->n_kv * n_indices >= ((int64_t)1 << 30))
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention_csr: n_kv x n_indices too large");
    if (!q || !kv_indptr || !context_lens || !out || (n_indices > 0 && !kv_indices))
        return fail(PKV_EINVAL, "paged_decode_attention_csr: NULL device pointer");
    if (((uintptr_t)q | (uintptr_t)out) & 15u)
        return fail(PKV_EINVAL, "paged_decode_attention_csr: q and out must be 16-byte aligned");
    if (((uintptr_t)kv_indptr | (uintptr_t)kv_indices | (uintptr_t)context_lens) & 3u)
        return fail(PKV_EINVAL, "paged_decode_attention_csr: indptr, indices and lengths must be 4-byte aligned");
    if (!pool->scales_set && pool->dtype != PKV_BF16)
        return fail(PKV_EINVAL, "paged_decode_attention_csr: quantised pool needs its scales first");

    DecodeArgs a;
    a.num_blocks = pool->num_blocks;
    a.n_kv = pool->n_kv;
    a.n_q = n_q;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = kv_indices;
    // W only sizes the grid and the workspace here: batch x W bounds the blocks
    a.W = (int)std::max<int64_t>(1, (n_indices + batch - 1) / batch);
    a.indptr = kv_indptr;
    a.n_indices = n_indices;
    a.context_lens = context_lens;
    a.batch = batch;
    a.qscale = scale * kLog2e;
    a.scales = pool->scales;
    a.k_params = pool->k_params;
    a.i4_entries = pool->dtype == PKV_INT4 ? static_cast<const uint8_t *>(pool->k) : nullptr;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.ws_ml = nullptr;
    a.ws_o = nullptr;
    a.slice_blocks = pool->partition_tokens / kBlockSize;
    a.err = pool->err;
    a.k_new = a.v_new = nullptr;
    a.k_pool = nullptr;
    a.skip_blocks = 0;
    a.n_pre = 0;
    a.pre_base = 0;
    return dispatch_kv(pool, a, G, static_cast<cudaStream_t>(stream));
}

namespace pkv {

// ---------------------------------------------------------------------------
// Fused step: append each sequence's newest token and decode, one launch
// ---------------------------------------------------------------------------

template <int D, int G, int KV>
static pkv_status launch_step(pkv_pool *pool, DecodeArgs a, cudaStream_t s)
{
    using C = Cfg<D, G, KV>;
    int grid = 0;
    size_t smem = 0;
    pkv_status st = decode_grid<D, G, KV, true>(pool, a.batch, a.W, &grid, &smem);
    if (st != PKV_OK) return st;
    const WsLayout L = ws_layout(a.n_q, a.n_kv, D, max_slots(pool, a.batch, a.n_kv, a.W, grid * C::NW));
    st = ensure_workspace(pool, L.total);
    if (st != PKV_OK) return st;
    bind_workspace(a, static_cast<uint8_t *>(pool->ws), L);
    LaunchScope ls(pool, kDecode, s);
    cudaError_t e = launch_pdl(decode_kernel<D, G, KV, true>, dim3(grid), dim3(C::kThreads), smem, s, pool->tm_entry,
                               a);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, "decode step launch");
    return launch_merge<D, G>(pool, a, grid * C::NW, s);
}

template <int D, int KV>
static pkv_status dispatch_step(pkv_pool *pool, const DecodeArgs &a, int G, cudaStream_t s)
{
    switch (G) {
    case 1: return launch_step<D, 1, KV>(pool, a, s);
    case 2: return launch_step<D, 2, KV>(pool, a, s);
    case 4: return launch_step<D, 4, KV>(pool, a, s);
    case 8: return launch_step<D, 8, KV>(pool, a, s);
    }
    return fail(PKV_EUNSUPPORTED, "decode step: group size %d unsupported (1, 2, 4 or 8)", G);
}

pkv_status check_step_args(const pkv_pool *pool, const char *who, int n_q, int max_blocks_per_seq, int batch,
                           float scale)
{
    if (!pool) return fail(PKV_EINVAL, "%s: NULL pool", who);
    if (batch < 0) return fail(PKV_EINVAL, "%s: batch < 0", who);
    if (n_q <= 0 || n_q % pool->n_kv)
        return fail(PKV_EINVAL, "%s: n_q %d is not a positive multiple of n_kv %d", who, n_q, pool->n_kv);
    const int G = n_q / pool->n_kv;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PKV_EUNSUPPORTED, "%s: n_q / n_kv = %d unsupported (1, 2, 4, 8)", who, G);
    if (max_blocks_per_seq <= 0 || max_blocks_per_seq > (1 << 24))
        return fail(PKV_EINVAL, "%s: max_blocks_per_seq %d out of range", who, max_blocks_per_seq);
    if (!isfinite(scale)) return fail(PKV_EINVAL, "%s: scale is not finite", who);
    if (batch > kMaxBatch) return fail(PKV_EUNSUPPORTED, "%s: batch %d > %d", who, batch, kMaxBatch);
    if ((int64_t)batch * pool->n_kv * max_blocks_per_seq >= ((int64_t)1 << 30))
        return fail(PKV_EUNSUPPORTED, "%s: batch x n_kv x max_blocks_per_seq too large", who);
    if (pool->dtype != PKV_BF16 && !pool->scales_set)
        return fail(PKV_EINVAL, "%s: quantised pool needs its scales first (kv_pool_set_fp8_scales or "
                    "kv_pool_set_int4_key_params)", who);
    return PKV_OK;
}

static pkv_status step_device(pkv_pool *pool, const void *q, const void *k_new, const void *v_new, int n_q,
                              const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                              int batch, float scale, void *out, cudaStream_t s)
{
    const int G = n_q / pool->n_kv;
    DecodeArgs a;
    a.num_blocks = pool->num_blocks;
    a.n_kv = pool->n_kv;
    a.n_q = n_q;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.W = max_blocks_per_seq;
    a.indptr = nullptr;
    a.n_indices = 0;
    a.context_lens = context_lens;
    a.batch = batch;
    a.qscale = scale * kLog2e;
    a.scales = pool->scales;
    a.k_params = pool->k_params;
    a.i4_entries = pool->dtype == PKV_INT4 ? static_cast<const uint8_t *>(pool->k) : nullptr;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.ws_ml = nullptr;
    a.ws_o = nullptr;
    a.slice_blocks = pool->partition_tokens / kBlockSize;
    a.err = pool->err;
    a.k_new = a.v_new = nullptr;
    a.k_pool = nullptr;
    a.skip_blocks = 0;
    a.n_pre = 0;
    a.pre_base = 0;
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.k_pool = static_cast<uint8_t *>(pool->k);
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    if (pool->dtype == PKV_INT4) {  // 4-bit pools: the append kernel (it finds the slots), then decode
        pkv_status st = append_step_int4(pool, k_new, v_new, block_tables, max_blocks_per_seq, context_lens,
                                         batch, s);
        if (st != PKV_OK) return st;
        a.k_new = a.v_new = nullptr;
        a.k_pool = nullptr;
        return dispatch_kv(pool, a, G, s);
    }
    if (pool->d_head == 128) return fp8 ? dispatch_step<128, true>(pool, a, G, s) : dispatch_step<128, false>(pool, a, G, s);
    return fp8 ? dispatch_step<64, true>(pool, a, G, s) : dispatch_step<64, false>(pool, a, G, s);
}

}  // namespace pkv

extern "C" pkv_status paged_decode_step(pkv_pool *pool, const void *q, const void *k_new, const void *v_new,
                                        int32_t n_q, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                        const int32_t *context_lens, int32_t batch, float scale, void *out,
                                        void *stream)
{
    pkv_status st = check_step_args(pool, "paged_decode_step", n_q, max_blocks_per_seq, batch, scale);
    if (st != PKV_OK || batch == 0) return st;
    if (!q || !k_new || !v_new || !block_tables || !context_lens || !out)
        return fail(PKV_EINVAL, "paged_decode_step: NULL device pointer");
    if (((uintptr_t)q | (uintptr_t)out | (uintptr_t)k_new | (uintptr_t)v_new) & 15u)
        return fail(PKV_EINVAL, "paged_decode_step: q, k_new, v_new and out must be 16-byte aligned");
    if (((uintptr_t)block_tables | (uintptr_t)context_lens) & 3u)
        return fail(PKV_EINVAL, "paged_decode_step: tables and lengths must be 4-byte aligned");
    return step_device(pool, q, k_new, v_new, n_q, block_tables, max_blocks_per_seq, context_lens, batch, scale,
                       out, static_cast<cudaStream_t>(stream));
}

namespace pkv {

// Host-memory gather for paged_decode_step_host: the step's inputs are read
// straight from pinned host memory (through its device mapping, over the
// CPU-GPU link) into the device staging area by one kernel, instead of one
// copy-engine transfer per array.
struct HostGather {
    const uint8_t *src[5];  // device addresses of mapped host buffers
    uint8_t *dst[5];
    int64_t bytes[5];
    int n;
};

__global__ void __launch_bounds__(256) host_gather_kernel(HostGather g)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int i = 0; i < g.n; ++i) {
        const uint8_t *src = g.src[i];
        uint8_t *dst = g.dst[i];
        const int64_t n = g.bytes[i];
        if ((((uintptr_t)src | (uintptr_t)dst | (uintptr_t)n) & 15u) == 0) {
            for (int64_t k = t0; k < n / 16; k += stride)
                reinterpret_cast<uint4 *>(dst)[k] = reinterpret_cast<const uint4 *>(src)[k];
        } else if ((((uintptr_t)src | (uintptr_t)dst | (uintptr_t)n) & 3u) == 0) {
            for (int64_t k = t0; k < n / 4; k += stride)
                reinterpret_cast<uint32_t *>(dst)[k] = reinterpret_cast<const uint32_t *>(src)[k];
        } else {
            for (int64_t k = t0; k < n; k += stride) dst[k] = src[k];
        }
    }
}

}  // namespace pkv

extern "C" pkv_status paged_decode_step_host(pkv_pool *pool, const void *q_host, const void *k_new_host,
                                             const void *v_new_host, int32_t n_q, const int32_t *block_tables_host,
                                             int32_t max_blocks_per_seq, const int32_t *context_lens_host,
                                             int32_t batch, float scale, void *out_host, void *stream)
{
    pkv_status st = check_step_args(pool, "paged_decode_step_host", n_q, max_blocks_per_seq, batch, scale);
    if (st != PKV_OK || batch == 0) return st;
    if (!q_host || !k_new_host || !v_new_host || !block_tables_host || !context_lens_host || !out_host)
        return fail(PKV_EINVAL, "paged_decode_step_host: NULL host pointer");
    const size_t D = pool->d_head;
    const size_t bq = (size_t)batch * n_q * D * 2, bkv = (size_t)batch * pool->n_kv * D * 2;
    const size_t bt = (size_t)batch * max_blocks_per_seq * 4, bl = (size_t)batch * 4;
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t o_q = 0, o_k = al(bq), o_v = o_k + al(bkv), o_t = o_v + al(bkv), o_l = o_t + al(bt),
                 o_o = o_l + al(bl), total = o_o + al(bq);
    st = ensure_staging(pool, total);
    if (st != PKV_OK) return st;
    uint8_t *d = static_cast<uint8_t *>(pool->stage);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const void *srcs[5] = {q_host, k_new_host, v_new_host, block_tables_host, context_lens_host};
    const size_t offs[5] = {o_q, o_k, o_v, o_t, o_l}, lens[5] = {bq, bkv, bkv, bt, bl};
    // Pinned buffers, no per-launch timing: the call's launches are replayed from a CUDA graph
    // captured on an earlier call with the same arguments (one submission instead of three).
    pkv_host_step_key key;
    {
        const void *ptrs[6] = {q_host, k_new_host, v_new_host, block_tables_host, context_lens_host, out_host};
        for (int i = 0; i < 6; ++i) key.ptr[i] = ptrs[i];
        key.n_q = n_q;
        key.W = max_blocks_per_seq;
        key.batch = batch;
        key.partition_tokens = pool->partition_tokens;
        memcpy(&key.scale_bits, &scale, 4);
        key.stage = pool->stage;
        key.ws = pool->ws;
        key.ws_bytes = pool->ws_bytes;
        key.stream = stream;
    }
    if (pool->host_graph && !pool->timing && key == pool->host_key) {
        cudaError_t e = cudaGraphLaunch(pool->host_graph, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "paged_decode_step_host: graph replay");
        return PKV_OK;
    }
    // Pinned (mapped) inputs: one gather kernel reads them all; otherwise one copy each.
    HostGather g = {};
    g.n = 5;
    bool mapped = true;
    for (int i = 0; i < 5 && mapped; ++i) {
        g.src[i] = static_cast<const uint8_t *>(mapped_host_ptr(srcs[i]));
        g.dst[i] = d + offs[i];
        g.bytes[i] = (int64_t)lens[i];
        mapped = g.src[i] != nullptr;
    }
    const int64_t units = (int64_t)(bq + 2 * bkv + bt + bl) / 16;
    const int ggrid = (int)std::max<int64_t>(1, std::min<int64_t>(2 * std::max(1, pool->num_sms), (units + 255) / 256));
    // Pinned (mapped), 16-byte aligned output: the kernels write it directly; otherwise staged and copied.
    void *out_dev = mapped_host_ptr(out_host);
    const bool direct_out = out_dev && ((uintptr_t)out_dev & 15u) == 0;
    // Mapped inputs aligned as the kernels read them (16 bytes for q and the new rows, 4 for the
    // tables and lengths): the step's kernels read them in place over the CPU-GPU link, no gather.
    const bool direct_in = mapped && direct_out &&
                           (((uintptr_t)g.src[0] | (uintptr_t)g.src[1] | (uintptr_t)g.src[2]) & 15u) == 0 &&
                           (((uintptr_t)g.src[3] | (uintptr_t)g.src[4]) & 3u) == 0;
    const uint8_t *in[5];
    for (int i = 0; i < 5; ++i) in[i] = direct_in ? g.src[i] : d + offs[i];
    auto run_step = [&](cudaStream_t ss) {
        return step_device(pool, in[0], in[1], in[2], n_q, reinterpret_cast<const int32_t *>(in[3]),
                           max_blocks_per_seq, reinterpret_cast<const int32_t *>(in[4]), batch, scale,
                           direct_out ? out_dev : d + o_o, ss);
    };
    if (direct_in) {
        // nothing to gather
    } else if (mapped) {
        host_gather_kernel<<<ggrid, 256, 0, s>>>(g);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "paged_decode_step_host: gather");
    } else {
        for (int i = 0; i < 5; ++i) {
            cudaError_t e = cudaMemcpyAsync(d + offs[i], srcs[i], lens[i], cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return cuda_fail(e, "paged_decode_step_host: copy in");
        }
    }
    st = run_step(s);
    if (st != PKV_OK) return st;
    cudaError_t e = direct_out ? cudaSuccess : cudaMemcpyAsync(out_host, d + o_o, bq, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "paged_decode_step_host: copy out");
    if (mapped && direct_out && !pool->timing) {
        // capture this call's launches for the next call with the same arguments (the buffers
        // have their final size now); a capture that fails only means no replay
        key.stage = pool->stage;
        key.ws = pool->ws;
        key.ws_bytes = pool->ws_bytes;
        if (!pool->capture_stream && cudaStreamCreateWithFlags(&pool->capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
            pool->capture_stream = nullptr;
            cudaGetLastError();
            return PKV_OK;
        }
        cudaStream_t cs = pool->capture_stream;
        cudaGraph_t graph = nullptr;
        bool ok = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
        if (ok) {
            if (!direct_in) {
                host_gather_kernel<<<ggrid, 256, 0, cs>>>(g);
                ok = cudaGetLastError() == cudaSuccess;
            }
            if (ok) ok = run_step(cs) == PKV_OK;
            const bool ended = cudaStreamEndCapture(cs, &graph) == cudaSuccess;
            ok = ok && ended && graph;
        }
        cudaGraphExec_t exec = nullptr;
        if (ok && cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess) {
            if (pool->host_graph) cudaGraphExecDestroy(pool->host_graph);
            pool->host_graph = exec;
            pool->host_key = key;
        }
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();  // a failed capture leaves no error behind for the caller
    }
    return PKV_OK;
}

namespace pkv {

// ---------------------------------------------------------------------------
// Cascade decode: a prefix shared by every sequence, read once
// ---------------------------------------------------------------------------
//
// "Memory Management in LLM Serving Systems", "Prefix sharing": storing a
// shared prefix once turns decode-time reads of n copies into one.  Stage 1
// is the decode kernel started past the prefix blocks (the sequences' own
// tails).  Stage 2 attends all batch x G query rows of each KV head to the
// prefix in one pass over its K and V tiles -- a dense contraction, run by
// the tcgen05 prefill kernel in partial mode -- and stores a (max, sum, O)
// partial per prefix chunk.  Stage 3, the merge kernel, combines the two.

// PKV_CASCADE_AUTO: whether the cascade pays for this prefix and batch, measured on GB300 (n_q 32,
// n_kv 8, d 128, tails of 0..1024 tokens, L2 warm and evicted).  bf16: from a 2048-token prefix
// with batch x prefix tokens >= 2^17 (1024-token prefixes run faster as plain decode at every
// batch up to 128, as do 2048 x 16 and 8192 x 8; 2048 x 64, 4096 x 32 and 8192 x 16 faster as the
// cascade).  FP8: plain decode pays its E4M3 conversions again on every re-read of the prefix, so
// the cascade pays earlier: from batch x prefix >= 2^16 with batch >= 64 (512 x 128, 1024 x 64),
// or >= 2^17 (1024 x 128: 47.6 against 65.8 us); 2048 x 32 and 4096 x 16 stay plain.
static bool cascade_pays(int dtype, int n_prefix_blocks, int batch)
{
    if (batch < 8) return false;
    const int64_t shared = (int64_t)n_prefix_blocks * kBlockSize * batch;
    if (dtype == PKV_FP8_E4M3) return shared >= (1 << 17) || (shared >= (1 << 16) && batch >= 64);
    return n_prefix_blocks >= 128 && shared >= (1 << 17);
}

template <int D, int G, int KV>
static pkv_status launch_prefix_decode(pkv_pool *pool, DecodeArgs a, const int32_t *prefix_blocks,
                                       int n_prefix_blocks, cudaStream_t s)
{
    using C = Cfg<D, G, KV>;
    int grid = 0;
    size_t smem = 0;
    pkv_status st = decode_grid<D, G, KV>(pool, a.batch, a.W, &grid, &smem);
    if (st != PKV_OK) return st;
    int chunk_blocks = 0, n_chunks = 0;
    prefix_stage_chunks(pool, a.batch, a.n_q, n_prefix_blocks, &chunk_blocks, &n_chunks);
    const int64_t tail_slots = max_slots(pool, a.batch, a.n_kv, a.W, grid * C::NW);
    const WsLayout L = ws_layout(a.n_q, a.n_kv, D, tail_slots + (int64_t)n_chunks * a.batch * a.n_kv);
    st = ensure_workspace(pool, L.total);
    if (st != PKV_OK) return st;
    bind_workspace(a, static_cast<uint8_t *>(pool->ws), L);
    a.skip_blocks = n_prefix_blocks;
    a.n_pre = n_chunks;
    a.pre_base = tail_slots;
    // Order: the tail decode, then the prefix stage (its CTAs take the SMs the
    // decode leaves as it finishes), then the merge.
    {
        LaunchScope ls(pool, kDecode, s);
        cudaError_t e = launch_pdl(decode_kernel<D, G, KV>, dim3(grid), dim3(C::kThreads), smem, s, pool->tm_entry,
                                   a);
        ls.done();
        if (e != cudaSuccess) return cuda_fail(e, "decode launch (cascade tail)");
    }
    st = launch_prefix_stage(pool, a.q, a.batch, a.n_q, prefix_blocks, n_prefix_blocks, chunk_blocks, n_chunks,
                             a.qscale, a.ws_ml, a.ws_o, tail_slots, s);
    if (st != PKV_OK) return st;
    return launch_merge<D, G>(pool, a, grid * C::NW, s);
}

template <int D, int KV>
static pkv_status dispatch_prefix(pkv_pool *pool, const DecodeArgs &a, int G, const int32_t *pb, int npb, cudaStream_t s)
{
    switch (G) {
    case 1: return launch_prefix_decode<D, 1, KV>(pool, a, pb, npb, s);
    case 2: return launch_prefix_decode<D, 2, KV>(pool, a, pb, npb, s);
    case 4: return launch_prefix_decode<D, 4, KV>(pool, a, pb, npb, s);
    case 8: return launch_prefix_decode<D, 8, KV>(pool, a, pb, npb, s);
    }
    return fail(PKV_EUNSUPPORTED, "cascade decode: group size %d unsupported (1, 2, 4 or 8)", G);
}

}  // namespace pkv

extern "C" pkv_status paged_decode_attention_prefix(pkv_pool *pool, const void *q, int32_t n_q,
                                                    const int32_t *prefix_blocks, int32_t n_prefix_blocks,
                                                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                    const int32_t *context_lens, int32_t batch, float scale,
                                                    void *out, void *stream)
{
    pkv_status st = check_step_args(pool, "paged_decode_attention_prefix", n_q, max_blocks_per_seq, batch, scale);
    if (st != PKV_OK || batch == 0) return st;
    if (pool->dtype == PKV_INT4)
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention_prefix: bf16 and FP8 pools only (not 4-bit)");
    if (n_prefix_blocks <= 0 || n_prefix_blocks > max_blocks_per_seq)
        return fail(PKV_EINVAL, "paged_decode_attention_prefix: n_prefix_blocks %d not in [1, max_blocks_per_seq]",
                    n_prefix_blocks);
    if (!q || !prefix_blocks || !block_tables || !context_lens || !out)
        return fail(PKV_EINVAL, "paged_decode_attention_prefix: NULL device pointer");
    if (((uintptr_t)q | (uintptr_t)out) & 15u)
        return fail(PKV_EINVAL, "paged_decode_attention_prefix: q and out must be 16-byte aligned");
    if (((uintptr_t)block_tables | (uintptr_t)context_lens | (uintptr_t)prefix_blocks) & 3u)
        return fail(PKV_EINVAL, "paged_decode_attention_prefix: tables and lengths must be 4-byte aligned");
    const int G = n_q / pool->n_kv;
    DecodeArgs a;
    a.num_blocks = pool->num_blocks;
    a.n_kv = pool->n_kv;
    a.n_q = n_q;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.W = max_blocks_per_seq;
    a.indptr = nullptr;
    a.n_indices = 0;
    a.context_lens = context_lens;
    a.batch = batch;
    a.qscale = scale * kLog2e;
    a.scales = pool->scales;
    a.k_params = pool->k_params;
    a.i4_entries = pool->dtype == PKV_INT4 ? static_cast<const uint8_t *>(pool->k) : nullptr;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.ws_ml = nullptr;
    a.ws_o = nullptr;
    a.slice_blocks = pool->partition_tokens / kBlockSize;
    a.err = pool->err;
    a.k_new = a.v_new = nullptr;
    a.k_pool = nullptr;
    a.skip_blocks = 0;
    a.n_pre = 0;
    a.pre_base = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Cascade or plain decode: with a short prefix the plain kernel's re-reads of it come
    // from L2 and cost less than the cascade's prefix stage and merge.
    const bool cascade = pool->cascade_mode == PKV_CASCADE_ALWAYS ||
                         (pool->cascade_mode == PKV_CASCADE_AUTO && cascade_pays(pool->dtype, n_prefix_blocks, batch));
    if (!cascade) return dispatch_kv(pool, a, G, s);
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    if (pool->d_head == 128)
        return fp8 ? dispatch_prefix<128, kKvFp8>(pool, a, G, prefix_blocks, n_prefix_blocks, s)
                   : dispatch_prefix<128, kKvBf16>(pool, a, G, prefix_blocks, n_prefix_blocks, s);
    return fp8 ? dispatch_prefix<64, kKvFp8>(pool, a, G, prefix_blocks, n_prefix_blocks, s)
               : dispatch_prefix<64, kKvBf16>(pool, a, G, prefix_blocks, n_prefix_blocks, s);
}

// ---------------------------------------------------------------------------
// Decode without allocation
//
// paged_decode_attention grows a workspace with cudaMalloc the first time a
// call needs more.  Some callers cannot allocate at that point: a serving
// engine that hands nearly all free HBM to its KV pool at start-up (as the
// memory-budget discussion of the pages describes engines doing) may have no
// room left, and cudaMalloc/cudaFree can synchronise the whole device, which
// a caller interleaving other streams' work cannot afford in its decode loop.
// paged_decode_attention_noalloc runs the same kernel with its scratch in a
// fixed, file-scope device array instead, so it never allocates.
// ---------------------------------------------------------------------------

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace pkv {

// In host code the array's name is only a host-side stand-in, never a device
// address: the address comes from cudaGetSymbolAddress, in the context that
// is current.  kv_pool_create calls this and keeps the result in the pool.
pkv_status noalloc_scratch_address(void **out)
{
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
    *out = ptr;
    return PKV_OK;
}

template <int D, int G, int KV>
static pkv_status launch_decode_noalloc(pkv_pool *pool, DecodeArgs a, uint8_t *scratch, cudaStream_t s)
{
    using C = Cfg<D, G, KV>;
    int grid = 0;
    size_t smem = 0;
    pkv_status st = decode_grid<D, G, KV>(pool, a.batch, a.W, &grid, &smem);
    if (st != PKV_OK) return st;
    const WsLayout L = ws_layout(a.n_q, a.n_kv, D, max_slots(pool, a.batch, a.n_kv, a.W, grid * C::NW));
    if (L.total > kNoAllocScratchBytes)
        return fail(PKV_ERANGE,
                    "paged_decode_attention_noalloc: this call needs %zu bytes of scratch but the static array "
                    "holds %zu; use paged_decode_attention (it grows a workspace) or a smaller batch",
                    L.total, kNoAllocScratchBytes);
    // The array keeps the previous call's contents; nothing in this layout
    // needs to start at zero (every partial is written before it is read).
    bind_workspace(a, scratch, L);
    LaunchScope ls(pool, kDecode, s);
    cudaError_t e = launch_pdl(decode_kernel<D, G, KV>, dim3(grid), dim3(C::kThreads), smem, s, pool->tm_entry,
                               a);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, "decode launch (noalloc)");
    return launch_merge<D, G>(pool, a, grid * C::NW, s);
}

template <int D, int KV>
static pkv_status dispatch_g_noalloc(pkv_pool *pool, const DecodeArgs &a, int G, uint8_t *scratch, cudaStream_t s)
{
    switch (G) {
    case 1: return launch_decode_noalloc<D, 1, KV>(pool, a, scratch, s);
    case 2: return launch_decode_noalloc<D, 2, KV>(pool, a, scratch, s);
    case 4: return launch_decode_noalloc<D, 4, KV>(pool, a, scratch, s);
    case 8: return launch_decode_noalloc<D, 8, KV>(pool, a, scratch, s);
    }
    return fail(PKV_EUNSUPPORTED, "decode: group size %d unsupported (1, 2, 4 or 8)", G);
}

}  // namespace pkv

extern "C" pkv_status paged_decode_attention_noalloc(pkv_pool *pool, const void *q, int32_t n_q,
                                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                     const int32_t *context_lens, int32_t batch, float scale,
                                                     void *out, void *stream)
{
    if (!pool) return fail(PKV_EINVAL, "paged_decode_attention_noalloc: NULL pool");
    if (batch < 0) return fail(PKV_EINVAL, "paged_decode_attention_noalloc: batch < 0");
    if (n_q <= 0 || n_q % pool->n_kv)
        return fail(PKV_EINVAL, "paged_decode_attention_noalloc: n_q %d is not a positive multiple of n_kv %d", n_q,
                    pool->n_kv);
    const int G = n_q / pool->n_kv;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention_noalloc: n_q / n_kv = %d unsupported (1, 2, 4, 8)", G);
    if (max_blocks_per_seq <= 0 || max_blocks_per_seq > (1 << 24))
        return fail(PKV_EINVAL, "paged_decode_attention_noalloc: max_blocks_per_seq %d out of range",
                    max_blocks_per_seq);
    if (!isfinite(scale)) return fail(PKV_EINVAL, "paged_decode_attention_noalloc: scale is not finite");
    if (batch == 0) return PKV_OK;
    if (batch > kMaxBatch)
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention_noalloc: batch %d > %d", batch, kMaxBatch);
    if ((int64_t)batch * pool->n_kv * max_blocks_per_seq >= ((int64_t)1 << 30))
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention_noalloc: batch x n_kv x max_blocks_per_seq too large");
    if (!q || !block_tables || !context_lens || !out)
        return fail(PKV_EINVAL, "paged_decode_attention_noalloc: NULL device pointer");
    if (((uintptr_t)q | (uintptr_t)out) & 15u)
        return fail(PKV_EINVAL, "paged_decode_attention_noalloc: q and out must be 16-byte aligned");
    if (((uintptr_t)block_tables | (uintptr_t)context_lens) & 3u)
        return fail(PKV_EINVAL, "paged_decode_attention_noalloc: tables and lengths must be 4-byte aligned");
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    if (!pool->scales_set && pool->dtype != PKV_BF16)
        return fail(PKV_EINVAL, "paged_decode_attention_noalloc: quantised pool needs its scales first");
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(e, "paged_decode_attention_noalloc: cudaGetDevice");
    if (cur != pool->device)
        return fail(PKV_EINVAL, "paged_decode_attention_noalloc: make the pool's device (%d) current, not %d",
                    pool->device, cur);
    void *scratch = pool->noalloc_scratch;  // looked up when the pool was created
    if (!scratch) return fail(PKV_ECUDA, "paged_decode_attention_noalloc: the pool has no scratch address");

    DecodeArgs a;
    a.num_blocks = pool->num_blocks;
    a.n_kv = pool->n_kv;
    a.n_q = n_q;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.W = max_blocks_per_seq;
    a.indptr = nullptr;
    a.n_indices = 0;
    a.context_lens = context_lens;
    a.batch = batch;
    a.qscale = scale * kLog2e;
    a.scales = pool->scales;
    a.k_params = pool->k_params;
    a.i4_entries = pool->dtype == PKV_INT4 ? static_cast<const uint8_t *>(pool->k) : nullptr;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.ws_ml = nullptr;
    a.ws_o = nullptr;
    a.slice_blocks = pool->partition_tokens / kBlockSize;
    a.err = pool->err;
    a.k_new = a.v_new = nullptr;
    a.k_pool = nullptr;
    a.skip_blocks = 0;
    a.n_pre = 0;
    a.pre_base = 0;
    uint8_t *sp = static_cast<uint8_t *>(scratch);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pool->d_head == 128)
        return pool->dtype == PKV_INT4 ? dispatch_g_noalloc<128, kKvInt4>(pool, a, G, sp, s)
               : fp8                   ? dispatch_g_noalloc<128, kKvFp8>(pool, a, G, sp, s)
                                       : dispatch_g_noalloc<128, kKvBf16>(pool, a, G, sp, s);
    return pool->dtype == PKV_INT4 ? dispatch_g_noalloc<64, kKvInt4>(pool, a, G, sp, s)
           : fp8                   ? dispatch_g_noalloc<64, kKvFp8>(pool, a, G, sp, s)
                                   : dispatch_g_noalloc<64, kKvBf16>(pool, a, G, sp, s);
}
