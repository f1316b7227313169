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
//     time share a few sequences' K/V in L2.  Row tiles go in pairs: CTAs 2i
//     and 2i + 1 take the two tiles of pair i, i + grid / 2, ..., so both
//     stream the same K/V tiles at about the same time (the second read comes
//     from L2).  Each CTA copies every tile it uses into its own shared
//     memory; nothing is shared between CTAs.  Every warp walks the list
//     itself from the chunk lengths (a window of 32 sequences held in
//     registers), so no role hands tiles to another.
//   * warp 8 streams Q (one 3-D TMA box per 64 columns) and the K tiles of
//     128 keys (8 blocks of 16 tokens, one 2-D TMA box per block and 64
//     columns) into a two-stage ring; warp 9 streams the V tiles likewise.
//     A missing block or an out-of-range block id loads a box past the end of
//     the pool (zero filled) and is masked out of the scores.
//   * warp 10 issues S = Q K^T for step j into one of two S accumulators in
//     tensor memory (128 fp32 columns each); warp 11 issues O_h += P_h V_h
//     for each key half h of a step as soon as that half's P is in tensor
//     memory, so the tensor cores compute the next scores while the softmax
//     warps work on the current ones.
//   * warps 0-7 run the softmax: warp w owns TMEM lanes (rows) 32 (w & 3) ..
//     + 31 and keys 64 (w >> 2) .. + 63 of every step.  Each key half of a
//     row keeps its own online softmax in the exp2 domain (reference maximum,
//     row sum, and its own accumulator O_h in tensor memory), so the two warps
//     of a lane quarter never wait for each other inside a tile.  The
//     reference maximum is raised lazily (O_h read, scaled and written back
//     only when a half's maximum grows by more than 2^8), so P stays at most
//     256 and almost every step skips the rescale.  P is rounded to bf16 for
//     the MMA, written over the half's scores, and the row sum adds the
//     rounded values, so the result is exactly a convex combination of the V
//     rows with the weights the MMA used.  At the tile's end the two warps of
//     a lane quarter swap (reference maximum, row sum) through shared memory,
//     combine O = (2^(m_0 - m) O_0 + 2^(m_1 - m) O_1) / l and store bf16.
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
constexpr int kSoftmaxWarps = 8;        // two per TMEM lane quarter: each takes half of a row's keys
constexpr int kKWarp = 8, kVWarp = 9, kQkWarp = 10, kPvWarp = 11;
constexpr int kThreads = 12 * 32;
constexpr float kRescaleSlack = 8.0f;    // log2 of the largest P value allowed before O is rescaled
// Tensor memory: S0 at 0, S1 at 128 (fp32 scores of a step), then one O
// accumulator per key half (O0 at 256, O1 at 256 + D).  A key half's P (bf16
// pairs: column j holds keys 2j, 2j + 1 of the half) is written over the first
// 32 columns of that half's own scores.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr int kKStages = 2, kVStages = 2;
constexpr uint32_t kHalf = 128 * 128;    // bytes of one 64-column half of a 128-row tile

struct Args {
    const int32_t *qo_indptr;  // [batch + 1]
    const int32_t *block_tables;
    int W;
    const int32_t *context_lens;
    // partial mode (the cascade's prefix stage): the "sequences" are chunks of
    // a block list shared by every sequence; each chunk's rows are all batch x
    // G query rows of a KV head; no causal mask; (m, l, O) partials out
    const int32_t *shared_blocks;
    int n_shared_blocks, chunk_blocks, n_chunks;
    float2 *ws_ml;             // [slot][G] (reference max, row sum)
    float *ws_o;               // [slot][G][D] unnormalised O
    int64_t pre_base;          // slot of (chunk c, sequence b, KV head g): pre_base + (c * batch + b) * n_kv + g
    int batch, n_q, n_kv;
    int64_t num_blocks;
    int64_t n_rows;            // rows of q and out: stores past them are skipped (an inconsistent indptr)
    int oob_row;               // a row index past the end of the pool's entry rows (zero-filled box)
    float qscale;              // scale * log2(e)
    const float *scales;       // FP8 pools: [2 * n_kv] fp32, K scales then V scales
    __nv_bfloat16 *out;        // [rows][n_q][D]
    unsigned *err;
};

template <int D>
struct Layout {
    static constexpr uint32_t QT = kRows * D * 2;        // one Q tile
    static constexpr uint32_t KT = kKeys * D * 2;        // one K (or V) step
    static constexpr uint32_t kQ = 0;                    // 2 Q buffers
    static constexpr uint32_t kK = kQ + 2 * QT;          // K stages
    static constexpr uint32_t kV = kK + kKStages * KT;   // V stages
    static constexpr uint32_t kOut = kV + kVStages * KT;  // the finished tile, staged for coalesced stores
    static constexpr uint32_t kBar = kOut + QT;
    // P_FULL and O_DONE: one per key half; DRAIN: one per issuer; PAIR: one per lane quarter
    enum { Q_FULL = 0, Q_FREE = 2, K_FULL = 4, K_EMPTY = 4 + kKStages, V_FULL = 4 + 2 * kKStages,
           V_EMPTY = V_FULL + kVStages, S_FULL = V_EMPTY + kVStages, S_FREE = S_FULL + 2, P_FULL = S_FREE + 2,
           O_DONE = P_FULL + 2, DRAIN = O_DONE + 2, OUT_FULL = DRAIN + 2, OUT_FREE = OUT_FULL + 1,
           PAIR = OUT_FREE + 1,
           // FP8 pools: the copies of Q, K and V complete on these; the producers convert
           // the landed bytes to f16 in place and then complete Q_FULL, K_FULL, V_FULL
           Q_RAW = PAIR + 4, K_RAW = Q_RAW + 2, V_RAW = K_RAW + kKStages, NBARS = V_RAW + kVStages };
    static constexpr uint32_t kTmemSlot = kBar + NBARS * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    // a tile's end: each key half's (reference maximum as bf16 bits, row sum) per row, for the other half
    static constexpr uint32_t kXm = (kAbort + 4 + 15) / 16 * 16;  // [2 halves][kRows] uint16
    static constexpr uint32_t kXl = kXm + 2 * kRows * 2;          // [2 halves][kRows] float
    static constexpr uint32_t kEnd = kXl + 2 * kRows * 4;
    static constexpr size_t bytes = 1024 + kEnd;
    static_assert(bytes <= 232448, "shared memory beyond the 227 KiB a CTA may use");
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

// Instruction descriptor, kind::f16: bf16 (f16 = false) or f16 (f16 = true)
// A and B, f32 accumulator, M x N, A K-major, B K-major (b_mn = 0) or
// MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, int b_mn, bool f16 = false)
{
    const uint32_t ab = f16 ? 0u : 1u;  // operand format: 0 f16, 1 bf16
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// A from tensor memory (M rows in lanes, K packed along columns), B from shared memory.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
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

// acc += the two bf16 halves of `pk` (each widened exactly, added in fp32).
__device__ __forceinline__ void add_bf16x2_to(float &acc, uint32_t pk)
{
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %0, hi, %0;\n\t}"
        : "+f"(acc)
        : "r"(pk));
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (a.x b.x + c.x, a.y b.y + c.y), each rounded as fmaf, in one paired instruction
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// acc += the two f16 halves of `pk` (each widened exactly, added in fp32).
__device__ __forceinline__ void add_f16x2_to(float &acc, uint32_t pk)
{
    asm("{\n\t.reg .b16 lo, hi;\n\t.reg .f32 a, b;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "cvt.f32.f16 a, lo;\n\tcvt.f32.f16 b, hi;\n\tadd.rn.f32 %0, a, %0;\n\tadd.rn.f32 %0, b, %0;\n\t}"
        : "+f"(acc)
        : "r"(pk));
}

// P as the operand the P V product takes: bf16 pairs, or f16 pairs for FP8 pools
// (whose MMAs run in f16); the row sum adds the rounded values.
template <bool F16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi)
{
    return F16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

template <bool F16>
__device__ __forceinline__ void add_p_to(float &acc, uint32_t pk)
{
    if constexpr (F16) add_f16x2_to(acc, pk);
    else add_bf16x2_to(acc, pk);
}

// ------------------------------------------------------------- FP8 pools: E4M3 -> f16 in shared memory

// Four E4M3 bytes -> two f16x2 words (bytes 0, 1 -> lo; bytes 2, 3 -> hi); exact.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t &lo, uint32_t &hi)
{
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// One step's K (or V) tile of an FP8 pool, converted in place by one warp.
// The copies put the 128 E4M3 rows (row r = key r of the step, D bytes, the
// pool's TMA swizzle: 16-byte chunk c of row r at chunk c ^ (r & 7) for
// 128-byte rows, c ^ ((r >> 1) & 3) for 64-byte rows) in the upper half of
// the stage; the f16 tile goes where the bf16 copies would have put it: per
// 64-column half, row r at r * 128 bytes, 16-byte chunk j at j ^ (r & 7).
// Rows are read before any lane writes (warp-synchronous) and taken in
// increasing order, so no write reaches an E4M3 row still to be read: for
// D = 128 the second half's row r is exactly E4M3 row r (so two warps may
// convert disjoint row ranges at the same time); for D = 64 the f16 row r
// covers E4M3 rows 2r - 128 and 2r - 127, both at most r (one warp, all rows).
// D = 128: rows [row0, row0 + rows), rows a multiple of 16.
template <int D>
__device__ __forceinline__ void convert_kv_f16(uint8_t *stage, int lane, int row0 = 0, int rows = kKeys)
{
    constexpr uint32_t KT = kKeys * D * 2;
    const uint32_t out = smem_u32(stage), in = out + KT / 2;
    if constexpr (D == 128) {
        // lane: row 4 i + lane / 8 (four iterations at a time), E4M3 chunk c = lane % 8 (columns 16 c .. + 15)
        constexpr int U = 4;
        const int c = lane & 7;
#pragma unroll 1
        for (int i = row0 / 4; i < (row0 + rows) / 4; i += U) {
            uint4 x[U];
            int r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                r[u] = 4 * (i + u) + (lane >> 3);
                x[u] = lds128(in + r[u] * 128 + ((c ^ (r[u] & 7)) << 4));
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < U; ++u) {
                uint4 lo, hi;
                e4m3x4_to_f16x4(x[u].x, lo.x, lo.y);
                e4m3x4_to_f16x4(x[u].y, lo.z, lo.w);
                e4m3x4_to_f16x4(x[u].z, hi.x, hi.y);
                e4m3x4_to_f16x4(x[u].w, hi.z, hi.w);
                const uint32_t row = out + (c >> 2) * kHalf + r[u] * 128;
                const int j = 2 * (c & 3);
                sts128(row + ((j ^ (r[u] & 7)) << 4), lo);
                sts128(row + (((j + 1) ^ (r[u] & 7)) << 4), hi);
            }
            __syncwarp();
        }
    } else {
        // lane: row 8 i + lane / 4 (four iterations at a time), E4M3 chunk c = lane % 4
        constexpr int U = 4;
        const int c = lane & 3;
#pragma unroll 1
        for (int i = 0; i < kKeys / 8; i += U) {
            uint4 x[U];
            int r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                r[u] = 8 * (i + u) + (lane >> 2);
                x[u] = lds128(in + r[u] * 64 + ((c ^ ((r[u] >> 1) & 3)) << 4));
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < U; ++u) {
                uint4 lo, hi;
                e4m3x4_to_f16x4(x[u].x, lo.x, lo.y);
                e4m3x4_to_f16x4(x[u].y, lo.z, lo.w);
                e4m3x4_to_f16x4(x[u].z, hi.x, hi.y);
                e4m3x4_to_f16x4(x[u].w, hi.z, hi.w);
                const uint32_t row = out + r[u] * 128;
                const int j = 2 * c;
                sts128(row + ((j ^ (r[u] & 7)) << 4), lo);
                sts128(row + (((j + 1) ^ (r[u] & 7)) << 4), hi);
            }
            __syncwarp();
        }
    }
}

// A Q tile (bf16, as the copy left it) -> f16 in place, element by element
// (exact for |q| in f16's normal range; larger values overflow f16).
template <int D>
__device__ __forceinline__ void convert_q_f16(uint8_t *qbuf, int lane)
{
    constexpr uint32_t QT = kRows * D * 2;
    const uint32_t base = smem_u32(qbuf);
#pragma unroll 4
    for (uint32_t off = 16u * lane; off < QT; off += 16u * 32) {
        uint4 v = lds128(base + off);
        uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = bf16x2_to_f32x2(w[k]);
            w[k] = pack_f16x2(f.x, f.y);
        }
        sts128(base + off, v);
    }
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
    int wb = 0;     // first sequence of the window
    int wbase = 0;  // pairs before sequence wb
    int incl = 0, tot = 0;
    int ph = 0, row0 = 0, T = 0, C = 0;  // this lane's sequence: pairs per KV head, rows, context
};

template <int G, bool PARTIAL>
__device__ __forceinline__ int n_items(const Args &a)
{
    return PARTIAL ? a.n_chunks : a.batch;
}

template <int G, bool PARTIAL>
__device__ __forceinline__ void load_window(Walker &w, const Args &a, int lane)
{
    const int bl = w.wb + lane;
    w.row0 = w.T = w.C = w.ph = 0;
    if (bl < n_items<G, PARTIAL>(a)) {
        if (PARTIAL) {  // chunk bl of the shared blocks: every sequence's query rows
            w.row0 = 0;
            w.T = a.batch;
            w.C = min(a.chunk_blocks, a.n_shared_blocks - bl * a.chunk_blocks) * kBlockSize;
        } else {
            w.row0 = a.qo_indptr[bl];
            w.T = a.qo_indptr[bl + 1] - w.row0;
            w.C = a.context_lens[bl];
        }
        if (w.T > 0) w.ph = ((w.T * G + kRows - 1) / kRows + 1) / 2;
    }
    int x = w.ph * a.n_kv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    w.incl = x;
    w.tot = __shfl_sync(kFull, x, 31);
}

// Pair x of the list of row-tile pairs; this CTA (`rank` = its index within
// the pair) takes row tile 2 i + rank of the pair's (sequence, KV head), i the
// pair's index there (past the last row tile when the count is odd: no rows
// and no steps).  The CTA streams the blocks its own last row reaches.  False
// past the list's end.  Warp-wide, uniform result.
template <int G, bool PARTIAL>
__device__ __forceinline__ bool find_tile(Walker &w, const Args &a, int x, int rank, Tile &t, int lane)
{
    while (x >= w.wbase + w.tot) {
        if (w.wb + 32 >= n_items<G, PARTIAL>(a)) return false;
        w.wbase += w.tot;
        w.wb += 32;
        load_window<G, PARTIAL>(w, a, lane);
    }
    const unsigned hit = __ballot_sync(kFull, w.wbase + w.incl > x);
    const int l = __ffs(hit) - 1;
    const int ph = __shfl_sync(kFull, w.ph, l);
    const int before = __shfl_sync(kFull, w.incl - w.ph * a.n_kv, l);
    t.b = w.wb + l;
    t.row0 = __shfl_sync(kFull, w.row0, l);
    t.T = __shfl_sync(kFull, w.T, l);
    int C = __shfl_sync(kFull, w.C, l);
    const int within = x - w.wbase - before;
    t.g = within / ph;
    const int pair_rt0 = 2 * (within - t.g * ph) * kRows;
    t.rt0 = pair_rt0 + rank * kRows;
    t.R = t.T * G;
    if (PARTIAL) {  // whole blocks, all visible to every row
        t.C = C;
        t.bad_ctx = false;
        t.n_blocks = C / kBlockSize;
        t.n_steps = (t.n_blocks + kStepBlocks - 1) / kStepBlocks;
        return true;
    }
    const int cap = a.W * kBlockSize;
    t.bad_ctx = C < t.T || C > cap;
    if (t.bad_ctx) C = max(t.T, min(C, cap));
    t.C = C;
    if (C > cap) {  // a chunk longer than the whole table: nothing sensible to attend to
        t.n_blocks = t.n_steps = 0;
        return true;
    }
    if (t.rt0 >= t.R) {  // the second tile of a pair with an odd tile count: no rows
        t.n_blocks = t.n_steps = 0;
        return true;
    }
    const int last_row = min(t.R, t.rt0 + kRows) - 1;
    t.n_blocks = (C - t.T + last_row / G) / kBlockSize + 1;
    t.n_steps = (t.n_blocks + kStepBlocks - 1) / kStepBlocks;
    return true;
}

// The block list a tile streams: its sequence's table row, or its chunk of the shared blocks.
template <bool PARTIAL>
__device__ __forceinline__ const int32_t *tile_blocks(const Args &a, const Tile &t)
{
    return PARTIAL ? a.shared_blocks + (int64_t)t.b * a.chunk_blocks : a.block_tables + (int64_t)t.b * a.W;
}

__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity)
{
    return __all_sync(kFull, mbar_wait_bounded(bar, parity));
}

// ------------------------------------------------------------- the kernel

template <int D, int G, bool PARTIAL, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv, Args a)
{
    using L = Layout<D>;
    constexpr int NH = D / 64 > 0 ? D / 64 : 1;  // 64-column halves of a row
    extern __shared__ __align__(1024) uint8_t tc_smem[];
    uint8_t *sm = tc_smem + ((1024u - (smem_u32(tc_smem) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kBar);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kAbort);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)(blockIdx.x & 1);  // which tile of a pair
    // FP8 pools with D = 128: each K (V) stage is widened to f16 half by the K (V) producer
    // warp (rows 0..63, one step behind its copies) and half by the warp that issues the MMAs
    // reading it (rows 64..127, just before it issues them)
    constexpr bool kSplitConv = F8 && D == 128;

    if (tid == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_kv);
        for (int i = 0; i < L::NBARS; ++i) {
            const bool by_warps = i == L::OUT_FULL || i == L::OUT_FREE;
            const bool by_half = i == L::P_FULL || i == L::P_FULL + 1;  // the four warps of a key half
            const bool by_pair = i >= L::PAIR && i < L::PAIR + 4;  // the two warps of a lane quarter
            // FP8, D = 128: a K or V stage is converted half by its producer, half by its MMA warp
            const bool by_conv = kSplitConv && ((i >= L::K_FULL && i < L::K_FULL + kKStages) ||
                                                (i >= L::V_FULL && i < L::V_FULL + kVStages));
            mbar_init(&bar[i], by_warps ? kSoftmaxWarps : by_half ? kSoftmaxWarps / 2 : (by_pair || by_conv) ? 2 : 1);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kQkWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(sm + L::kTmemSlot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();  // the barriers and the tensor-memory address are visible to every warp
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + L::kTmemSlot);
    // queries, tables and the appended chunk may come from the previous kernel.  In
    // partial mode the previous kernel is the cascade's tail decode, whose output this
    // kernel does not read: it waits at its end instead, so that the merge launched after
    // it sees both.
    if (!PARTIAL) griddep_wait();
    griddep_launch_dependents();

    auto set_abort = [&]() {
        if (lane == 0) {
            atomicOr(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    };

    Walker wk;
    load_window<G, PARTIAL>(wk, a, lane);

    if (warp == kKWarp || warp == kVWarp) {
        // ---------------------------------------------------------- producers
        const bool is_k = warp == kKWarp;
        const int NS = is_k ? kKStages : kVStages;
        const CUtensorMap *map = &tm_kv;  // 16-row boxes over the entries' key and value rows
        const uint32_t ring = is_k ? L::kK : L::kV;
        uint64_t *full = &bar[is_k ? L::K_FULL : L::V_FULL];
        uint64_t *empty = &bar[is_k ? L::K_EMPTY : L::V_EMPTY];
        // FP8 pools: the copies complete on `raw` instead; the E4M3 tile lands in the upper
        // half of its stage and this warp converts it to f16 in place one step later (after
        // issuing the next step's copies, so their latency overlaps the conversion), then
        // completes `full`.  The K warp converts each tile's Q (bf16 -> f16) with the tile's
        // first K step.
        uint64_t *raw = &bar[is_k ? L::K_RAW : L::V_RAW];
        uint64_t *land = F8 ? raw : full;
        const int qland = F8 ? L::Q_RAW : L::Q_FULL;
        const uint64_t policy = l2_policy_evict_normal();
        int gs = 0, qi = 0;
        int pend = -1, pend_q = -1;  // FP8: the step awaiting conversion, and the Q load to convert before it
        bool ok = true;
        [[maybe_unused]] auto convert_pending = [&]() -> bool {
            if (pend_q >= 0) {
                const int qb = pend_q & 1;
                if (!wait_all(&bar[L::Q_RAW + qb], (pend_q >> 1) & 1)) return false;
                convert_q_f16<D>(sm + L::kQ + qb * L::QT, lane);
                fence_proxy_async_smem();  // the MMAs read the converted tile through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[L::Q_FULL + qb]);
            }
            const int st = pend % NS;
            if (!wait_all(&raw[st], (pend / NS) & 1)) return false;
            if constexpr (kSplitConv) convert_kv_f16<D>(sm + ring + st * L::KT, lane, 0, kKeys / 2);
            else convert_kv_f16<D>(sm + ring + st * L::KT, lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[st]);
            return true;
        };
        for (int x = blockIdx.x / 2; ok; x += gridDim.x / 2) {
            Tile t;
            if (!find_tile<G, PARTIAL>(wk, a, x, rank, t, lane)) break;
            if (t.n_steps == 0) continue;
            if (*abort_flag) break;
            const int32_t *trow = tile_blocks<PARTIAL>(a, t);
            // block ids (lanes 0..7) one step ahead of the copies: the table read is off the refill path
            int nxt = lane < kStepBlocks && lane < t.n_blocks ? trow[lane] : -1;
            int q_load = -1;
            if (is_k) {  // this tile's queries into Q buffer qi & 1
                const int qb = qi & 1;
                if (qi >= 2 && !(ok = wait_all(&bar[L::Q_FREE + qb], ((qi >> 1) + 1) & 1))) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar[qland + qb], L::QT);
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        tma_load_3d(sm + L::kQ + qb * L::QT + h * kHalf, &tm_q, 64 * h, t.g * G,
                                    t.row0 + t.rt0 / G, &bar[qland + qb], policy);
                }
                q_load = qi;
                ++qi;
            }
            for (int s = 0; s < t.n_steps; ++s, ++gs) {
                const int cur = nxt;
                const int nb = (s + 1) * kStepBlocks + lane;
                if (s + 1 < t.n_steps) nxt = lane < kStepBlocks && nb < t.n_blocks ? trow[nb] : -1;
                const int st = gs % NS, use = gs / NS;
                if (use > 0 && !(ok = wait_all(&empty[st], (use - 1) & 1))) break;
                const bool present = lane < kStepBlocks && s * kStepBlocks + lane < t.n_blocks;
                const bool valid = present && cur >= 0 && cur < a.num_blocks;
                if (present && !valid && is_k) atomicOr(a.err, PKV_DEVERR_BLOCK_RANGE);
                if (lane == 0) mbar_arrive_expect_tx(&land[st], F8 ? L::KT / 2 : L::KT);
                __syncwarp();
                if (lane < kStepBlocks) {  // lane k copies block k of the step
                    // the block's key rows open its (block, KV head) entry, its value rows follow
                    const int y = valid ? (int)((cur * (int64_t)a.n_kv + t.g) * 2 * kBlockSize + (is_k ? 0 : kBlockSize))
                                        : a.oob_row;
                    if constexpr (F8) {  // one box per block: 16 E4M3 rows of D bytes
                        tma_load_2d(sm + ring + st * L::KT + L::KT / 2 + lane * (kBlockSize * D), map, 0, y,
                                    &raw[st], policy);
                    } else {
                        uint8_t *dst = sm + ring + st * L::KT + lane * (kBlockSize * 128);
#pragma unroll
                        for (int h = 0; h < NH; ++h) tma_load_2d(dst + h * kHalf, map, 64 * h, y, &full[st], policy);
                    }
                }
                if constexpr (F8) {
                    if (pend >= 0 && !(ok = convert_pending())) break;
                    pend = gs;
                    pend_q = s == 0 ? q_load : -1;
                }
            }
        }
        if constexpr (F8) {
            if (ok && pend >= 0 && !*abort_flag) ok = convert_pending();
        }
        // copies still in flight (after an abort) land before the CTA exits
        for (int j = 1; j <= NS && gs - j >= 0; ++j) {
            const int g2 = gs - j;
            mbar_wait_bounded(&land[g2 % NS], (g2 / NS) & 1);
        }
        if (is_k && qi > 0) mbar_wait_bounded(&bar[qland + ((qi - 1) & 1)], ((qi - 1) >> 1) & 1);
        if (is_k && qi > 1) mbar_wait_bounded(&bar[qland + ((qi - 2) & 1)], ((qi - 2) >> 1) & 1);
        if (!ok) set_abort();
    } else if (warp == kQkWarp || warp == kPvWarp) {
        // ---------------------------------------------------------- MMA issue
        // Two issuing warps, so that neither's waits and commits hold up the
        // other: S = Q K^T runs up to two steps ahead (as far as the two S
        // accumulators allow), O += P V starts as soon as a step's P is in
        // tensor memory.  Each warp commits, and finally drains, its own MMAs.
        const bool is_qk = warp == kQkWarp;
        constexpr uint32_t idesc_qk = mma_idesc(kRows, kKeys, 0, F8);
        constexpr uint32_t idesc_pv = mma_idesc(kRows, D, 1, F8);
        const uint32_t base = smem_u32(sm);
        int gs = 0, qi = 0;
        bool ok = true;
        for (int x = blockIdx.x / 2; ok; x += gridDim.x / 2) {
            Tile t;
            if (!find_tile<G, PARTIAL>(wk, a, x, rank, t, lane)) break;
            if (t.n_steps == 0) continue;
            if (*abort_flag) break;
            const int qb = qi & 1;
            if (is_qk && !(ok = wait_all(&bar[L::Q_FULL + qb], (qi >> 1) & 1))) break;
            for (int s = 0; s < t.n_steps && ok; ++s, ++gs) {
                if (is_qk) {
                    const int st = gs & 1, kst = gs % kKStages;
                    if constexpr (kSplitConv) {  // rows 64..127 of this K stage
                        if (!(ok = wait_all(&bar[L::K_RAW + kst], (gs / kKStages) & 1))) break;
                        convert_kv_f16<D>(sm + L::kK + kst * L::KT, lane, kKeys / 2, kKeys / 2);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[L::K_FULL + kst]);
                    }
                    if (!(ok = wait_all(&bar[L::K_FULL + kst], (gs / kKStages) & 1))) break;
                    if (gs >= 2 && !(ok = wait_all(&bar[L::S_FREE + st], ((gs >> 1) + 1) & 1))) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t qbase = base + L::kQ + qb * L::QT, kbase = base + L::kK + kst * L::KT;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                            umma(tmem + st * kKeys, smem_desc(qbase + off, 16, 1024),
                                 smem_desc(kbase + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        umma_commit(&bar[L::S_FULL + st]);
                        umma_commit(&bar[L::K_EMPTY + kst]);
                        if (s == t.n_steps - 1) umma_commit(&bar[L::Q_FREE + qb]);
                    }
                } else {
                    // O_h += P_h V_h for each key half h as soon as its P is in tensor memory; the
                    // step's S buffer (which holds the two P) is free once both have run
                    const int vst = gs % kVStages, st = gs & 1;
                    if constexpr (kSplitConv) {  // rows 64..127 of this V stage
                        if (!(ok = wait_all(&bar[L::V_RAW + vst], (gs / kVStages) & 1))) break;
                        convert_kv_f16<D>(sm + L::kV + vst * L::KT, lane, kKeys / 2, kKeys / 2);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[L::V_FULL + vst]);
                    }
                    if (!(ok = wait_all(&bar[L::V_FULL + vst], (gs / kVStages) & 1))) break;
                    const uint32_t vb = base + L::kV + vst * L::KT;
                    for (int h = 0; h < 2; ++h) {
                        if (!(ok = wait_all(&bar[L::P_FULL + h], gs & 1))) break;
                        tc_fence_after();
                        if (lane == 0) {
#pragma unroll
                            for (int kk = 0; kk < kKeys / 32; ++kk) {  // keys 64 h + 16 kk .. + 15
                                const uint32_t at = tmem + st * kKeys + h * (kKeys / 2) + 8 * kk;
                                const uint64_t bd = smem_desc(vb + (h * (kKeys / 32) + kk) * 2048, kHalf, 1024);
                                umma_ts(tmem + kColO + h * D, at, bd, idesc_pv, (s > 0 || kk > 0) ? 1u : 0u);
                            }
                            umma_commit(&bar[L::O_DONE + h]);
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    if (lane == 0) {
                        umma_commit(&bar[L::S_FREE + st]);
                        umma_commit(&bar[L::V_EMPTY + vst]);
                    }
                }
                __syncwarp();
            }
            ++qi;
        }
        // every MMA this warp issued has completed before the tensor memory is released
        uint64_t *drain = &bar[L::DRAIN + (is_qk ? 0 : 1)];
        if (lane == 0) umma_commit(drain);
        __syncwarp();
        mbar_wait_bounded(drain, 0);
        if (!ok) set_abort();
    } else {
        // ---------------------------------------------------------- softmax
        // warp w: TMEM lanes (rows) 32 (w & 3) .. + 31 and keys 64 (w >> 2) .. + 63 of every step.
        // The two key halves of a row run separate online softmaxes (each its own reference
        // maximum, row sum and O accumulator), so the two warps of a lane quarter never wait for
        // each other inside a tile; at the tile's end they combine the halves by log-sum-exp.
        constexpr int HK = kKeys / 2, HD = D / 2;
        const int quarter = warp & 3, ch = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint64_t *pair = &bar[L::PAIR + quarter];
        int pph = 0;              // completed phases of the pair barrier (two per tile)
        bool o_in_use = false;    // the partner may still read this half's O (previous tile)
        uint16_t *xm = reinterpret_cast<uint16_t *>(sm + L::kXm);
        float *xl = reinterpret_cast<float *>(sm + L::kXl);
        constexpr int QB = kStepBlocks / 2;  // blocks of a step in this warp's key half
        // this warp's block ids of step 0 of tile t (lanes 0..QB-1)
        auto first_ids = [&](const Tile &t) -> int {
            return lane < QB && ch * QB + lane < t.n_blocks ? tile_blocks<PARTIAL>(a, t)[ch * QB + lane] : -1;
        };
        int gs = 0, n_out = 0;  // steps so far, tiles written out so far
        bool ok = true;
        int x = blockIdx.x / 2;
        Tile t, tn;
        bool have = find_tile<G, PARTIAL>(wk, a, x, rank, t, lane);
        int nxt = have ? first_ids(t) : -1;
        while (have && ok) {
            // the next tile and its first block ids are found while this one runs
            const bool have_n = find_tile<G, PARTIAL>(wk, a, x + gridDim.x / 2, rank, tn, lane);
            if (t.bad_ctx && tid == 0 && t.rt0 == 0 && t.g == 0) atomicOr(a.err, PKV_DEVERR_CTX_RANGE);
            if (t.n_steps == 0 || *abort_flag) {
                if (*abort_flag) break;
                x += gridDim.x / 2;
                t = tn;
                have = have_n;
                nxt = have ? first_ids(t) : -1;
                continue;
            }
            const int r = t.rt0 + row;
            const int64_t orow_i = (int64_t)t.row0 + min(r, t.R - 1) / G;  // this row's query token
            const bool in_out = orow_i >= 0 && orow_i < a.n_rows;
            if (r < t.R && !in_out && ch == 0) atomicOr(a.err, PKV_DEVERR_CTX_RANGE);
            // this row's position: it sees keys 0 .. pos (every key of a shared chunk)
            const int pos = PARTIAL ? t.C - 1 : t.C - t.T + min(r, t.R - 1) / G;
            // FP8 pools: the K scale of this KV head folds into the score scale, the V scale
            // into the final normalisation
            const float qs = F8 ? a.qscale * a.scales[t.g] : a.qscale;
            const float vs = F8 ? a.scales[a.n_kv + t.g] : 1.0f;
            float mref = -INFINITY;  // this half's reference maximum: a bf16 value (sent exactly at the end)
            float l4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // this half's row sum of the bf16-rounded P
            // block ids of this warp's 4 blocks of the next step (lanes 0..3), read one step ahead
            // (for the last step: the next tile's first ids): the same validity test as the
            // producers, so a masked block is exactly a skipped one
            const int32_t *trow = tile_blocks<PARTIAL>(a, t);
            for (int s = 0; s < t.n_steps; ++s, ++gs) {
                const int cur = nxt;
                const int nb = (s + 1) * kStepBlocks + ch * QB + lane;
                if (s + 1 < t.n_steps) nxt = lane < QB && nb < t.n_blocks ? trow[nb] : -1;
                else nxt = have_n ? first_ids(tn) : -1;
                const uint32_t mask = __ballot_sync(kFull, lane < QB && cur >= 0 && cur < a.num_blocks) & ((1u << QB) - 1);
                const int sb = gs & 1;
                if (!(ok = wait_all(&bar[L::S_FULL + sb], (gs >> 1) & 1))) break;
                tc_fence_after();
                uint32_t sr[HK];
#pragma unroll
                for (int c = 0; c < HK / 32; ++c) tmem_ld32(tmem + lane_off + sb * kKeys + ch * HK + 32 * c, sr + 32 * c);
                tmem_wait_ld();

                const int key0 = s * kKeys + ch * HK;  // position of this warp's first key
                if (!(mask == (1u << QB) - 1 && key0 + HK - 1 <= pos)) {
#pragma unroll
                    for (int k = 0; k < HK; ++k) {
                        const bool vis = ((mask >> (k / kBlockSize)) & 1u) && key0 + k <= pos;
                        if (!vis) sr[k] = __float_as_uint(-INFINITY);
                    }
                }
                // row maximum of this half: 8 independent chains of 3-input maxima
                static_assert(HK == 64, "the max chains assume 64 keys per warp and step");
                float m4[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    auto v = [&](int t) { return __uint_as_float(sr[j + 8 * t]); };
                    m4[j] = fmaxf(fmax3(fmax3(fmax3(v(0), v(1), v(2)), v(3), v(4)), v(5), v(6)), v(7));
                }
                const float bm_half = fmax3(fmax3(m4[0], m4[1], m4[2]), fmax3(m4[3], m4[4], m4[5]),
                                            fmaxf(m4[6], m4[7]));
                const float bms = bm_half * qs;
                const bool resc = bms > mref + kRescaleSlack;
                float alpha = 1.0f;
                if (resc) {
                    const float mnew = __bfloat162float(__float2bfloat16_ru(bms));  // >= bms
                    alpha = ex2(mref - mnew);  // 0 when mref is -inf
                    mref = mnew;
#pragma unroll
                    for (int i = 0; i < 4; ++i) l4[i] *= alpha;
                }
                const float nm = mref == -INFINITY ? 0.0f : -mref;
                uint32_t pk[HK / 2];
#pragma unroll
                for (int i = 0; i < HK / 2; ++i) {
                    const float2 x = ffma2(make_float2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])),
                                           make_float2(qs, qs), make_float2(nm, nm));
                    pk[i] = pack_p<F8>(ex2(x.x), ex2(x.y));
                    add_p_to<F8>(l4[i & 3], pk[i]);
                }
                if (s > 0) {
                    // this half's previous O += P V has finished (waited at every step and at the
                    // tile's end, so the parity waits follow the barrier's phases one by one); only
                    // then may O be rescaled
                    if (!(ok = wait_all(&bar[L::O_DONE + ch], (gs - 1) & 1))) break;
                    if (__any_sync(kFull, resc)) {
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tmem + lane_off + kColO + ch * D + 32 * c, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(tmem + lane_off + kColO + ch * D + 32 * c, o);
                        }
                    }
                }
                // P over this half's scores of the step (already read)
                tmem_st32(tmem + lane_off + sb * kKeys + ch * HK, pk);
                tmem_wait_st();
                if (o_in_use) {  // the partner has read this half's O of the previous tile
                    if (!(ok = wait_all(pair, pph & 1))) break;
                    ++pph;
                    o_in_use = false;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[L::P_FULL + ch]);
            }
            if (!ok) break;
            // epilogue: combine the two halves (log-sum-exp), then O / l for this tile's rows,
            // this warp's half of the columns
            if (!(ok = wait_all(&bar[L::O_DONE + ch], (gs - 1) & 1))) break;
            const float l_half = (l4[0] + l4[1]) + (l4[2] + l4[3]);
            xm[ch * kRows + row] = __bfloat16_as_ushort(__float2bfloat16_rn(mref));  // exact: a bf16 value
            xl[ch * kRows + row] = l_half;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pair);
            if (!(ok = wait_all(pair, pph & 1))) break;  // both halves' O and (m, l) are final
            ++pph;
            tc_fence_after();
            const float m_ot = __bfloat162float(__ushort_as_bfloat16(xm[(ch ^ 1) * kRows + row]));
            const float l_ot = xl[(ch ^ 1) * kRows + row];
            const float mrow = fmaxf(mref, m_ot);  // the row's reference maximum
            const float f_me = mref == -INFINITY ? 0.0f : ex2(mref - mrow);
            const float f_ot = m_ot == -INFINITY ? 0.0f : ex2(m_ot - mrow);
            const float l = l_half * f_me + l_ot * f_ot;
            const float inv = l > 0.0f ? vs / l : 0.0f;
            // partial mode: O carries the V scale (the merge divides by the summed l only)
            const float pv = PARTIAL ? vs : 1.0f;
            const float f0 = (ch == 0 ? f_me : f_ot) * pv, f1 = (ch == 0 ? f_ot : f_me) * pv;
            // columns ch * HD + 32 c .. + 31 of the row's O = f0 O0 + f1 O1
            auto load_o = [&](int c, uint32_t (&o)[32]) {
                uint32_t o1[32];
                tmem_ld32(tmem + lane_off + kColO + ch * HD + 32 * c, o);
                tmem_ld32(tmem + lane_off + kColO + D + ch * HD + 32 * c, o1);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] = __float_as_uint(fmaf(f1, __uint_as_float(o1[i]), f0 * __uint_as_float(o[i])));
            };
            if (PARTIAL) {  // (m, l, O) of this row for the merge, this warp's half of O
                const bool rv = r < t.R;
                const int64_t slot = a.pre_base + ((int64_t)t.b * a.batch + (rv ? r / G : 0)) * a.n_kv + t.g;
                float *wo = a.ws_o + (slot * G + r % G) * D + ch * HD;
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    load_o(c, o);
                    if (rv) {
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            *reinterpret_cast<float4 *>(wo + 32 * c + 4 * q4) =
                                make_float4(__uint_as_float(o[4 * q4]), __uint_as_float(o[4 * q4 + 1]),
                                            __uint_as_float(o[4 * q4 + 2]), __uint_as_float(o[4 * q4 + 3]));
                    }
                }
                if (rv && ch == 0) a.ws_ml[slot * G + r % G] = make_float2(mrow, l);
            } else if (t.rt0 < t.R) {  // (a pair's second tile may hold no rows)
                // this warp's half row of O / l into the staging tile, 16-byte chunks
                // swizzled within each 128-byte half row (conflict-free writes and reads)
                constexpr int RB = D * 2;  // bytes of an output row
                uint8_t *stage = sm + L::kOut;
                if (n_out > 0 && !(ok = wait_all(&bar[L::OUT_FREE], (n_out - 1) & 1))) break;
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    load_o(c, o);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
                        const int chunk = (ch * HD + 32 * c + 8 * q4) / 8;  // 16-byte chunk of the row
                        *reinterpret_cast<uint4 *>(stage + row * RB + ((chunk >> 3) << 7) +
                                                   (((chunk & 7) ^ (row & 7)) << 4)) = w;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[L::OUT_FULL]);
                if (!(ok = wait_all(&bar[L::OUT_FULL], n_out & 1))) break;
                // coalesced: consecutive threads store consecutive 16-byte chunks of a row
                constexpr int CPR = RB / 16;  // chunks per row
                for (int i = warp * 32 + lane; i < kRows * CPR; i += kSoftmaxWarps * 32) {
                    const int rr = i / CPR, chunk = i % CPR;
                    const int rg = t.rt0 + rr;
                    const int64_t tok = (int64_t)t.row0 + rg / G;
                    if (rg < t.R && tok >= 0 && tok < a.n_rows) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(stage + rr * RB + ((chunk >> 3) << 7) +
                                                                         (((chunk & 7) ^ (rr & 7)) << 4));
                        *reinterpret_cast<uint4 *>(a.out + (tok * a.n_q + t.g * G + rg % G) * D + chunk * 8) = w;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[L::OUT_FREE]);
                ++n_out;
            }
            // both halves' O of this tile are read: the partner's next P may let O += P V overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pair);
            o_in_use = true;
            x += gridDim.x / 2;
            t = tn;
            have = have_n;
        }
        if (!ok) set_abort();
    }

    tc_fence_before();
    __syncthreads();  // every role is done with the tensor memory
    tc_fence_after();
    if (PARTIAL) griddep_wait();
    if (warp == kQkWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// CTAs of the kernel that fit on the device at once (one per SM), rounded
// down to whole pairs.
template <int D, int G, bool PARTIAL, bool F8>
pkv_status setup(pkv_pool *pool, int *max_pairs)
{
    using L = Layout<D>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int occ = 0;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(prefill_tc_kernel<D, G, PARTIAL, F8>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
        if (attr_err == cudaSuccess)
            attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, prefill_tc_kernel<D, G, PARTIAL, F8>,
                                                                     kThreads, L::bytes);
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "prefill kernel attributes");
    if (occ < 1) return fail(PKV_ECUDA, "prefill: the kernel does not fit on an SM");
    *max_pairs = std::max(1, occ * pool->num_sms / 2);
    return PKV_OK;
}

// pairs: an upper bound on the row-tile pairs (the grid is at most two CTAs per pair).
template <int D, int G, bool PARTIAL, bool F8>
pkv_status launch(pkv_pool *pool, const void *q, int64_t n_rows, int n_q, int64_t pairs, const Args &a,
                  cudaStream_t s)
{
    using L = Layout<D>;
    int max_pairs = 0;
    pkv_status st = setup<D, G, PARTIAL, F8>(pool, &max_pairs);
    if (st != PKV_OK) return st;
    CUtensorMap tm_q;
    st = make_q_map(&tm_q, q, n_rows, n_q, D, G, kRows / G);
    if (st != PKV_OK) return st;
    const int grid = 2 * (int)std::min<int64_t>(pairs, max_pairs);
    LaunchScope ls(pool, PARTIAL ? kPrefix : kDecode, s);
    cudaError_t e = launch_pdl(prefill_tc_kernel<D, G, PARTIAL, F8>, dim3(grid), dim3(kThreads), L::bytes, s, tm_q,
                               pool->tm_block, a);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, PARTIAL ? "prefix stage launch" : "prefill launch");
    return PKV_OK;
}

template <int D, bool PARTIAL, bool F8>
pkv_status dispatch_g(pkv_pool *pool, const void *q, int64_t n_rows, int n_q, int G, int64_t pairs, const Args &a,
                      cudaStream_t s)
{
    switch (G) {
    case 1: return launch<D, 1, PARTIAL, F8>(pool, q, n_rows, n_q, pairs, a, s);
    case 2: return launch<D, 2, PARTIAL, F8>(pool, q, n_rows, n_q, pairs, a, s);
    case 4: return launch<D, 4, PARTIAL, F8>(pool, q, n_rows, n_q, pairs, a, s);
    case 8: return launch<D, 8, PARTIAL, F8>(pool, q, n_rows, n_q, pairs, a, s);
    }
    return fail(PKV_EUNSUPPORTED, "prefill: group size %d unsupported (1, 2, 4 or 8)", G);
}

// The launch for the pool's head size and KV type (bf16 or FP8 E4M3).
template <bool PARTIAL>
pkv_status dispatch(pkv_pool *pool, const void *q, int64_t n_rows, int n_q, int G, int64_t pairs, const Args &a,
                    cudaStream_t s)
{
    const bool f8 = pool->dtype == PKV_FP8_E4M3;
    if (pool->d_head == 128)
        return f8 ? dispatch_g<128, PARTIAL, true>(pool, q, n_rows, n_q, G, pairs, a, s)
                  : dispatch_g<128, PARTIAL, false>(pool, q, n_rows, n_q, G, pairs, a, s);
    return f8 ? dispatch_g<64, PARTIAL, true>(pool, q, n_rows, n_q, G, pairs, a, s)
              : dispatch_g<64, PARTIAL, false>(pool, q, n_rows, n_q, G, pairs, a, s);
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
    if (pool->dtype == PKV_INT4)
        return fail(PKV_EUNSUPPORTED, "paged_prefill_attention: bf16 and FP8 pools only (not 4-bit)");
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
    a.oob_row = (int)(pool->num_blocks * pool->n_kv * 2 * kBlockSize);
    a.qscale = scale * kLog2e;
    a.scales = pool->scales;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = pool->err;
    a.shared_blocks = nullptr;
    a.n_shared_blocks = a.chunk_blocks = a.n_chunks = 0;
    a.ws_ml = nullptr;
    a.ws_o = nullptr;
    a.pre_base = 0;
    const int G = n_q / pool->n_kv;
    // an upper bound on the row-tile pairs: every sequence may end with a partial tile
    const int64_t pairs = ((n_rows * G + kRows - 1) / kRows + batch) * pool->n_kv;
    if (pairs > INT32_MAX || n_rows * G > INT32_MAX)
        return fail(PKV_EUNSUPPORTED, "paged_prefill_attention: too many query rows");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dispatch<false>(pool, q, n_rows, n_q, G, pairs, a, s);
}

namespace pkv {

void prefix_stage_chunks(pkv_pool *pool, int batch, int n_q, int n_prefix_blocks, int *chunk_blocks, int *n_chunks)
{
    const int G = n_q / pool->n_kv;
    const int64_t pairs_per_chunk = (int64_t)pool->n_kv * ((((int64_t)batch * G + kRows - 1) / kRows + 1) / 2);
    // about one CTA pair per pair of SMs, and at least two steps of blocks per chunk
    const int64_t want = std::max<int64_t>(1, (pool->num_sms / 2) / std::max<int64_t>(1, pairs_per_chunk));
    const int64_t cap = std::max<int64_t>(1, (n_prefix_blocks + 2 * kStepBlocks - 1) / (2 * kStepBlocks));
    const int nc = (int)std::min(want, cap);
    *chunk_blocks = (n_prefix_blocks + nc - 1) / nc;
    *n_chunks = (n_prefix_blocks + *chunk_blocks - 1) / *chunk_blocks;
}

pkv_status launch_prefix_stage(pkv_pool *pool, const void *q, int batch, int n_q, const int32_t *prefix_blocks,
                               int n_prefix_blocks, int chunk_blocks, int n_chunks, float qscale, float2 *ws_ml,
                               float *ws_o,
                               int64_t pre_base, cudaStream_t s)
{
    const int G = n_q / pool->n_kv;
    Args a;
    a.qo_indptr = nullptr;
    a.block_tables = nullptr;
    a.W = 0;
    a.context_lens = nullptr;
    a.batch = batch;
    a.n_q = n_q;
    a.n_kv = pool->n_kv;
    a.num_blocks = pool->num_blocks;
    a.n_rows = batch;
    a.oob_row = (int)(pool->num_blocks * pool->n_kv * 2 * kBlockSize);
    a.qscale = qscale;
    a.scales = pool->scales;
    a.out = nullptr;
    a.err = pool->err;
    a.shared_blocks = prefix_blocks;
    a.n_shared_blocks = n_prefix_blocks;
    a.chunk_blocks = chunk_blocks;
    a.n_chunks = n_chunks;
    a.ws_ml = ws_ml;
    a.ws_o = ws_o;
    a.pre_base = pre_base;
    const int64_t pairs = (int64_t)a.n_chunks * pool->n_kv * ((((int64_t)batch * G + kRows - 1) / kRows + 1) / 2);
    return dispatch<true>(pool, q, batch, n_q, G, pairs, a, s);
}

}  // namespace pkv
