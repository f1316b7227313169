// Paged GQA decode attention: one new query token per sequence against its
// cached keys and values, read through the sequence's block table.
//
// What is computed ("The KV Cache from First Principles", "Implementation";
// "KV cache, PagedAttention and FlashAttention", Problems 4 and 5):
//   out[b][h] = sum_p softmax_p(scale * q[b][h] . K[p][g]) V[p][g],
//   g = h / (n_q / n_kv), p < context_len[b], K/V of position p in block
//   block_table[b][p / 16] at offset p % 16.
//
// How (GB300 design, see the file-level notes in the header):
//   * Work unit = (sequence, KV head, partition of `part_blocks` blocks).
//     Long sequences split across thread blocks ("Serving note" of Problem 5;
//     "Memory Management in LLM Serving Systems", FlashAttention-2: parallelise
//     over the sequence dimension).  A persistent grid of
//     (#SMs x resident CTAs) walks the units; the partition count of every
//     sequence comes from an in-kernel prefix sum over context_lens, so the
//     host never reads lengths and the call never synchronises.
//   * Each CTA has 4 warps.  Each warp owns a ring of shared-memory stages;
//     lane 0 fetches the (block, KV head) K tile and V tile of its next blocks
//     with 1-D bulk TMA copies (cp.async.bulk, evict-first L2 hint) that
//     complete on an mbarrier.  Every wait is bounded.
//   * All G query heads of the group are served from one read of each tile
//     ("Memory Management in LLM Serving Systems", FlashAttention: several
//     query heads against the same KV block cut KV reads by the group factor).
//   * Scores: each lane dots 8 elements of a key with the G query rows held
//     in registers, then a transpose-reduce over the key's lanes leaves one
//     (token, head) score per lane.  Online softmax in fp32 with exp2 (q is
//     pre-scaled by scale*log2 e): running max m and sum l per head, the
//     accumulator rescaled only when the max moves (Problem 5's recurrence;
//     FlashAttention-2's deferred 1/l).
//   * P.V: each lane owns D/32 output columns of all G heads.
//   * Unit end: the 4 warps' (m, l, o) merge in shared memory; a sequence with
//     one partition writes bf16 `out` directly, otherwise (m, l, o) go to the
//     workspace and merge_kernel combines partitions by log-sum-exp:
//     M = max m_p, L = sum 2^(m_p-M) l_p, out = sum 2^(m_p-M) o_p / L.
//   * FP8 KV: tiles are E4M3, converted in registers; the K scale is folded
//     into q and the V scale into the final normalisation.
#include <algorithm>
#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxBatch = 8192;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
    const uint8_t *k_pool, *v_pool;
    int64_t num_blocks;
    int n_kv, n_q;
    const __nv_bfloat16 *q;
    const int32_t *block_tables;
    int W;
    const int32_t *context_lens;
    int batch;
    float qscale;          // scale * log2(e)
    const float *scales;   // FP8: [2 * n_kv] (k then v)
    __nv_bfloat16 *out;
    int32_t *part_start;   // workspace [batch + 1]
    float2 *ws_ml;         // workspace [P][n_kv][G] (max in log2 units, sum)
    float *ws_o;           // workspace [P][n_kv][G][D], unnormalised
    int part_blocks;       // blocks per partition (multiple of kWarps)
    unsigned *err;
};

template <int D, int G, bool FP8>
struct Cfg {
    static constexpr int E = FP8 ? 1 : 2;
    static constexpr int kTileBytes = kBlockSize * D * E;   // one (block, head) tile
    static constexpr int kStageBytes = 2 * kTileBytes;      // K tile + V tile
    static constexpr int kStages = std::min(8, std::max(2, 16384 / kStageBytes));
    static constexpr int LPT = D / 8;        // lanes per key row in the score phase
    static constexpr int TPR = 32 / LPT;     // keys per round
    static constexpr int SPAN = LPT / G;     // lanes sharing one head after the halving
    static constexpr int DPL = D / 32;       // output columns per lane in the P.V phase
    // shared-memory layout (bytes)
    static constexpr int kRing = kWarps * kStages * kStageBytes;
    static constexpr int kBars = kRing;
    static constexpr int kPhys = kBars + kWarps * kStages * 8;
    static constexpr int kSp = kPhys + kWarps * kStages * 4;
    static constexpr int kMergeM = kSp + kWarps * kBlockSize * 8 * 4;
    static constexpr int kMergeL = kMergeM + kWarps * 8 * 4;
    static constexpr int kMergeO = kMergeL + kWarps * 8 * 4;
    static constexpr int kPartStart = kMergeO + kWarps * G * D * 4;
    static size_t smem_bytes(int batch) { return (size_t)kPartStart + 4 * (size_t)(batch + 1); }
    static_assert(G <= LPT, "group larger than lanes per key");
};

__device__ __forceinline__ int clamp_ctx(int c, int W, unsigned *err, bool report)
{
    const int cmax = W * kBlockSize;
    if (c < 0 || c > cmax) {
        if (report) atomicOr(err, PKV_DEVERR_CTX_RANGE);
        c = c < 0 ? 0 : cmax;
    }
    return c;
}

// Exclusive prefix sum of partitions per sequence into ps[0..batch].
__device__ void scan_partitions(const DecodeArgs &a, int32_t *ps)
{
    __shared__ int warp_tot[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int carry = 0;
    for (int base = 0; base < a.batch; base += kThreads) {
        const int b = base + tid;
        int n = 0;
        if (b < a.batch) {
            const int c = clamp_ctx(a.context_lens[b], a.W, a.err, blockIdx.x == 0);
            const int nblk = (c + kBlockSize - 1) / kBlockSize;
            n = (nblk + a.part_blocks - 1) / a.part_blocks;
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
        for (int w = 0; w < kWarps; ++w) {
            const int t = warp_tot[w];
            before += (w < warp) ? t : 0;
            tot += t;
        }
        if (b < a.batch) ps[b] = carry + before + x - n;
        carry += tot;
        __syncthreads();
    }
    if (tid == 0) ps[a.batch] = carry;
    __syncthreads();
}

struct Unit {
    int b, g, pidx, nparts, j0, j1, C;
};

__device__ __forceinline__ Unit decode_unit(int u, const DecodeArgs &a, const int32_t *ps)
{
    Unit r;
    r.pidx = u / a.n_kv;
    r.g = u - r.pidx * a.n_kv;
    int lo = 0, hi = a.batch - 1;  // largest b with ps[b] <= pidx
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ps[mid] <= r.pidx) lo = mid; else hi = mid - 1;
    }
    r.b = lo;
    r.nparts = ps[lo + 1] - ps[lo];
    r.C = clamp_ctx(a.context_lens[lo], a.W, a.err, false);
    const int nblk = (r.C + kBlockSize - 1) / kBlockSize;
    r.j0 = (r.pidx - ps[lo]) * a.part_blocks;
    r.j1 = min(r.j0 + a.part_blocks, nblk);
    return r;
}

// The sequence of (unit, block) items one warp consumes, in order.
struct Iter {
    int u, j, j1, b, g;
};

__device__ __forceinline__ bool iter_next(Iter &it, int warp, int total_units, const DecodeArgs &a,
                                          const int32_t *ps)
{
    it.j += kWarps;
    while (it.j >= it.j1) {
        it.u += gridDim.x;
        if (it.u >= total_units) return false;
        const Unit un = decode_unit(it.u, a, ps);
        it.b = un.b;
        it.g = un.g;
        it.j = un.j0 + warp;
        it.j1 = un.j1;
    }
    return true;
}

// 8 consecutive stored elements -> fp32.
template <bool FP8>
__device__ __forceinline__ void load8(const uint8_t *p, float (&f)[8])
{
    if constexpr (!FP8) {
        const uint4 r = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = bf16x2_to_f32x2(w[i]);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    } else {
        const uint2 r = *reinterpret_cast<const uint2 *>(p);
        const uint32_t w[2] = {r.x, r.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float2 lo = e4m3x2_to_f32x2(w[i] & 0xffffu);
            const float2 hi = e4m3x2_to_f32x2(w[i] >> 16);
            f[4 * i] = lo.x;
            f[4 * i + 1] = lo.y;
            f[4 * i + 2] = hi.x;
            f[4 * i + 3] = hi.y;
        }
    }
}

// N (= 2 or 4) consecutive stored elements -> fp32.
template <bool FP8, int N>
__device__ __forceinline__ void loadN(const uint8_t *p, float (&f)[N])
{
    if constexpr (!FP8) {
        if constexpr (N == 4) {
            const uint2 r = *reinterpret_cast<const uint2 *>(p);
            const float2 a = bf16x2_to_f32x2(r.x), b = bf16x2_to_f32x2(r.y);
            f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        } else {
            const float2 a = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t *>(p));
            f[0] = a.x; f[1] = a.y;
        }
    } else {
        if constexpr (N == 4) {
            const uint32_t r = *reinterpret_cast<const uint32_t *>(p);
            const float2 a = e4m3x2_to_f32x2(r & 0xffffu), b = e4m3x2_to_f32x2(r >> 16);
            f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        } else {
            const float2 a = e4m3x2_to_f32x2(*reinterpret_cast<const uint16_t *>(p));
            f[0] = a.x; f[1] = a.y;
        }
    }
}

// Halving steps of the transpose-reduce: N values per lane, exchanged across
// lane bit OFF; the upper lane keeps the upper half.  After log2(G) steps
// lane `sub` holds head sub / SPAN, summed over its partner lanes.
template <int N, int OFF, int G>
__device__ __forceinline__ void halve(float (&v)[G], int lane)
{
    if constexpr (N > 1) {
        const bool upper = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float send = upper ? v[i] : v[i + N / 2];
            const float keep = upper ? v[i + N / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, OFF);
        }
        halve<N / 2, OFF / 2, G>(v, lane);
    }
}

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeArgs a)
{
    using C = Cfg<D, G, FP8>;
    constexpr int S = C::kStages;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t *ring = smem + warp * S * C::kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBars) + warp * S;
    int *phys_st = reinterpret_cast<int *>(smem + C::kPhys) + warp * S;
    float *sp = reinterpret_cast<float *>(smem + C::kSp) + warp * kBlockSize * 8;
    float *merge_m = reinterpret_cast<float *>(smem + C::kMergeM);
    float *merge_l = reinterpret_cast<float *>(smem + C::kMergeL);
    float *merge_o = reinterpret_cast<float *>(smem + C::kMergeO);
    int32_t *ps = reinterpret_cast<int32_t *>(smem + C::kPartStart);

    if (tid == 0) {
        for (int i = 0; i < kWarps * S; ++i)
            mbar_init(reinterpret_cast<uint64_t *>(smem + C::kBars) + i, 1);
        fence_mbarrier_init();
    }
    scan_partitions(a, ps);  // ends with __syncthreads
    const int total_units = ps[a.batch] * a.n_kv;
    if (blockIdx.x == 0)
        for (int i = tid; i <= a.batch; i += kThreads) a.part_start[i] = ps[i];
    // Sequences with no cached tokens get a zero output row.
    for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
        if (ps[b + 1] != ps[b]) continue;
        uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t)b * a.n_q * D);
        for (int i = tid; i < a.n_q * D / 8; i += kThreads) o[i] = make_uint4(0, 0, 0, 0);
    }

    const uint64_t policy = l2_policy_evict_first();
    const int sub = lane % C::LPT, tsub = lane / C::LPT;  // score phase
    const int hl = lane & 7, tq = lane >> 3;              // softmax phase
    bool aborted = false;
    int drain_from = -1;  // first item whose copy may still be in flight after a timeout

    // Producer state (uniform across the warp; lane 0 issues).
    Iter pit;
    pit.u = blockIdx.x - gridDim.x;
    pit.j = 0;
    pit.j1 = 0;
    pit.b = pit.g = 0;
    bool prod_done = false;
    int n_issued = 0;
    auto issue = [&](int n) {
        const int st = n % S;
        if (lane == 0) {
            const int64_t phys = a.block_tables[(int64_t)pit.b * a.W + pit.j];
            const bool ok = phys >= 0 && phys < a.num_blocks;
            phys_st[st] = ok ? (int)phys : -1;
            if (ok) {
                const int64_t tile = (phys * a.n_kv + pit.g) * (int64_t)C::kTileBytes;
                uint8_t *dst = ring + st * C::kStageBytes;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[st], 2 * C::kTileBytes);
                bulk_g2s(dst, a.k_pool + tile, C::kTileBytes, &bars[st], policy);
                bulk_g2s(dst + C::kTileBytes, a.v_pool + tile, C::kTileBytes, &bars[st], policy);
            } else {
                atomicOr(a.err, PKV_DEVERR_BLOCK_RANGE);
                mbar_arrive(&bars[st]);
            }
        }
    };
    for (; n_issued < S; ++n_issued) {
        if (!iter_next(pit, warp, total_units, a, ps)) {
            prod_done = true;
            break;
        }
        issue(n_issued);
    }

    int consumed = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
        const Unit un = decode_unit(u, a, ps);
        // q rows of the group, pre-scaled so that scores come out in log2 units.
        const float qs = a.qscale * (FP8 ? a.scales[un.g] : 1.0f);
        float qf[G][8];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const uint4 r = ldg_nc_v4(a.q + ((int64_t)un.b * a.n_q + un.g * G + hh) * D + sub * 8);
            const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 x = bf16x2_to_f32x2(w[i]);
                qf[hh][2 * i] = x.x * qs;
                qf[hh][2 * i + 1] = x.y * qs;
            }
        }
        float acc[G][C::DPL];
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int i = 0; i < C::DPL; ++i) acc[hh][i] = 0.0f;
        float m_run = -INFINITY, l_run = 0.0f;  // per lane: head hl, tokens of quarter tq

        for (int j = un.j0 + warp; j < un.j1; j += kWarps) {
            const int st = consumed % S;
            const uint32_t parity = (uint32_t)(consumed / S) & 1u;
            if (!aborted) {
                const bool ok = mbar_wait_bounded(&bars[st], parity);
                aborted = __any_sync(kFull, !ok);
                if (aborted) {
                    drain_from = consumed;
                    if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
                }
            }
            if (!aborted && phys_st[st] >= 0) {
                const uint8_t *kt = ring + st * C::kStageBytes;
                const uint8_t *vt = kt + C::kTileBytes;
                const int nv = min(kBlockSize, un.C - j * kBlockSize);
                // ---- scores for the block's 16 keys x G heads ----
#pragma unroll
                for (int r = 0; r < kBlockSize / C::TPR; ++r) {
                    const int t = r * C::TPR + tsub;
                    float kf[8];
                    load8<FP8>(kt + (t * D + sub * 8) * C::E, kf);
                    float part[G];
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        float s = 0.0f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) s = fmaf(qf[hh][i], kf[i], s);
                        part[hh] = s;
                    }
                    halve<G, C::LPT / 2, G>(part, lane);
                    float x = part[0];
#pragma unroll
                    for (int off = C::SPAN / 2; off >= 1; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
                    if (sub % C::SPAN == 0) sp[t * 8 + sub / C::SPAN] = (t < nv) ? x : -INFINITY;
                }
                __syncwarp();
                // ---- online softmax update (lane: head hl, keys 4tq..4tq+3) ----
                float s4[4];
                float bm = -INFINITY;
                if (hl < G) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        s4[i] = sp[(tq * 4 + i) * 8 + hl];
                        bm = fmaxf(bm, s4[i]);
                    }
                }
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
                const float m_new = fmaxf(m_run, bm);
                float alpha = 1.0f;
                if (hl < G) {
                    float lsum = 0.0f;
                    if (m_new != -INFINITY) {
                        alpha = exp2f(m_run - m_new);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float p = exp2f(s4[i] - m_new);
                            sp[(tq * 4 + i) * 8 + hl] = p;
                            lsum += p;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) sp[(tq * 4 + i) * 8 + hl] = 0.0f;
                    }
                    l_run = l_run * alpha + lsum;
                    m_run = m_new;
                }
                __syncwarp();
                if (__any_sync(kFull, alpha != 1.0f)) {
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const float al = __shfl_sync(kFull, alpha, hh);
#pragma unroll
                        for (int i = 0; i < C::DPL; ++i) acc[hh][i] *= al;
                    }
                }
                // ---- P.V ----
#pragma unroll 4
                for (int t = 0; t < nv; ++t) {
                    float p[G];
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) p[hh] = sp[t * 8 + hh];
                    float vf[C::DPL];
                    loadN<FP8, C::DPL>(vt + (t * D + lane * C::DPL) * C::E, vf);
#pragma unroll
                    for (int hh = 0; hh < G; ++hh)
#pragma unroll
                        for (int i = 0; i < C::DPL; ++i) acc[hh][i] = fmaf(p[hh], vf[i], acc[hh][i]);
                }
            }
            __syncwarp();
            ++consumed;
            if (!prod_done && !aborted) {
                if (iter_next(pit, warp, total_units, a, ps)) {
                    issue(n_issued);
                    ++n_issued;
                } else {
                    prod_done = true;
                }
            }
        }

        // ---- merge the 4 warps' (m, l, o) for this unit ----
        float l_tot = l_run + __shfl_xor_sync(kFull, l_run, 8);
        l_tot += __shfl_xor_sync(kFull, l_tot, 16);
        if (lane < G) {
            merge_m[warp * 8 + lane] = m_run;
            merge_l[warp * 8 + lane] = l_tot;
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int i = 0; i < C::DPL; ++i) merge_o[(warp * G + hh) * D + lane * C::DPL + i] = acc[hh][i];
        __syncthreads();
        const float vs = FP8 ? a.scales[a.n_kv + un.g] : 1.0f;
        for (int idx = tid; idx < G * D; idx += kThreads) {
            const int hh = idx / D, d = idx - hh * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, merge_m[w * 8 + hh]);
            float L = 0.0f, o = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float sc = exp2f(merge_m[w * 8 + hh] - M);
                    L = fmaf(sc, merge_l[w * 8 + hh], L);
                    o = fmaf(sc, merge_o[(w * G + hh) * D + d], o);
                }
            }
            o *= vs;
            if (un.nparts == 1) {
                a.out[((int64_t)un.b * a.n_q + un.g * G + hh) * D + d] =
                    __float2bfloat16_rn(L > 0.0f ? o / L : 0.0f);
            } else {
                const int64_t r = ((int64_t)un.pidx * a.n_kv + un.g) * G + hh;
                a.ws_o[r * D + d] = o;
                if (d == 0) a.ws_ml[r] = make_float2(M, L);
            }
        }
        __syncthreads();
    }

    // Only after a timeout can copies still be in flight: wait for them
    // (bounded) before the CTA's shared memory goes away.
    if (drain_from >= 0)
        for (int k = drain_from; k < n_issued; ++k)
            mbar_wait_bounded(&bars[k % S], (uint32_t)(k / S) & 1u, 100000000ull);
}

struct MergeArgs {
    int batch, n_q, n_kv;
    const int32_t *part_start;
    const float2 *ws_ml;
    const float *ws_o;
    __nv_bfloat16 *out;
};

// One warp per (sequence, query head) with two or more partitions: lanes form
// 4 groups of 8; group k combines partitions k, k+4, ...; each lane owns D/8
// consecutive columns.  Log-sum-exp merge in log2 units.
template <int D, int G>
__global__ void __launch_bounds__(128) merge_kernel(MergeArgs a)
{
    constexpr int DPL = D / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    if (row >= a.batch * a.n_q) return;
    const int b = row / a.n_q, h = row - b * a.n_q;
    const int g = h / G, hh = h - g * G;
    const int p0 = a.part_start[b], np = a.part_start[b + 1] - p0;
    if (np <= 1) return;
    float M = -INFINITY;
    for (int p = lane; p < np; p += 32) M = fmaxf(M, a.ws_ml[((int64_t)(p0 + p) * a.n_kv + g) * G + hh].x);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    const int grp = lane >> 3, sl = lane & 7;
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.0f;
    float L = 0.0f;
#pragma unroll 2
    for (int p = grp; p < np; p += 4) {
        const int64_t r = ((int64_t)(p0 + p) * a.n_kv + g) * G + hh;
        const float2 ml = a.ws_ml[r];
        const float sc = (M == -INFINITY) ? 0.0f : exp2f(ml.x - M);
        L = fmaf(sc, ml.y, L);
        const float4 *src = reinterpret_cast<const float4 *>(a.ws_o + r * D + sl * DPL);
#pragma unroll
        for (int i = 0; i < DPL / 4; ++i) {
            const float4 x = src[i];
            acc[4 * i] = fmaf(sc, x.x, acc[4 * i]);
            acc[4 * i + 1] = fmaf(sc, x.y, acc[4 * i + 1]);
            acc[4 * i + 2] = fmaf(sc, x.z, acc[4 * i + 2]);
            acc[4 * i + 3] = fmaf(sc, x.w, acc[4 * i + 3]);
        }
    }
    L += __shfl_xor_sync(kFull, L, 8);
    L += __shfl_xor_sync(kFull, L, 16);
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
        acc[i] += __shfl_xor_sync(kFull, acc[i], 8);
        acc[i] += __shfl_xor_sync(kFull, acc[i], 16);
    }
    if (grp == 0) {
        __nv_bfloat16 *o = a.out + (int64_t)row * D + sl * DPL;
#pragma unroll
        for (int i = 0; i < DPL; i += 2) {
            const float x0 = L > 0.0f ? acc[i] / L : 0.0f;
            const float x1 = L > 0.0f ? acc[i + 1] / L : 0.0f;
            *reinterpret_cast<__nv_bfloat162 *>(o + i) = __floats2bfloat162_rn(x0, x1);
        }
    }
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t decode_workspace_bytes(int batch, int n_q, int n_kv, int d_head, int max_blocks_per_seq,
                              int partition_tokens)
{
    const int part_blocks = partition_tokens / kBlockSize;
    const int64_t nps = (max_blocks_per_seq + part_blocks - 1) / part_blocks;
    const int64_t P = (int64_t)batch * nps;
    const int G = n_q / n_kv;
    return align256(4 * (size_t)(batch + 1)) + align256(8 * (size_t)P * n_kv * G) +
           4 * (size_t)P * n_kv * G * d_head;
}

template <int D, int G, bool FP8>
static pkv_status launch_decode(pkv_pool *pool, const DecodeArgs &a, int nps, cudaStream_t s)
{
    using C = Cfg<D, G, FP8>;
    auto kern = decode_kernel<D, G, FP8>;
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
    const size_t smem = C::smem_bytes(a.batch);
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (occ < 1) return fail(PKV_EUNSUPPORTED, "decode: %zu bytes of shared memory do not fit", smem);
    const int64_t units_max = (int64_t)a.batch * nps * a.n_kv;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(units_max, (int64_t)pool->num_sms * occ));
    {
        LaunchScope ls(pool, kDecode, s);
        kern<<<(unsigned)grid, kThreads, smem, s>>>(a);
        e = cudaGetLastError();
        ls.done();
        if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    }
    if (nps > 1) {
        MergeArgs m;
        m.batch = a.batch;
        m.n_q = a.n_q;
        m.n_kv = a.n_kv;
        m.part_start = a.part_start;
        m.ws_ml = a.ws_ml;
        m.ws_o = a.ws_o;
        m.out = a.out;
        const int rows = a.batch * a.n_q;
        LaunchScope ls(pool, kMerge, s);
        merge_kernel<D, G><<<(rows + 3) / 4, 128, 0, s>>>(m);
        e = cudaGetLastError();
        ls.done();
        if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    }
    return PKV_OK;
}

template <int D, bool FP8>
static pkv_status dispatch_g(pkv_pool *pool, const DecodeArgs &a, int G, int nps, cudaStream_t s)
{
    switch (G) {
    case 1: return launch_decode<D, 1, FP8>(pool, a, nps, s);
    case 2: return launch_decode<D, 2, FP8>(pool, a, nps, s);
    case 4: return launch_decode<D, 4, FP8>(pool, a, nps, s);
    case 8: return launch_decode<D, 8, FP8>(pool, a, nps, s);
    }
    return fail(PKV_EUNSUPPORTED, "decode: group size %d unsupported (1, 2, 4 or 8)", G);
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
    if (!q || !block_tables || !context_lens || !out)
        return fail(PKV_EINVAL, "paged_decode_attention: NULL device pointer");
    if (((uintptr_t)q | (uintptr_t)out) & 15u)
        return fail(PKV_EINVAL, "paged_decode_attention: q and out must be 16-byte aligned");
    if (((uintptr_t)block_tables | (uintptr_t)context_lens) & 3u)
        return fail(PKV_EINVAL, "paged_decode_attention: tables and lengths must be 4-byte aligned");
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    if (fp8 && !pool->scales_set)
        return fail(PKV_EINVAL, "paged_decode_attention: FP8 pool needs kv_pool_set_fp8_scales first");

    const int part_blocks = pool->partition_tokens / kBlockSize;
    const int nps = (max_blocks_per_seq + part_blocks - 1) / part_blocks;
    if ((int64_t)batch * nps * pool->n_kv * G >= ((int64_t)1 << 31))
        return fail(PKV_EUNSUPPORTED, "paged_decode_attention: too many partitions; raise the partition size");
    const size_t need = decode_workspace_bytes(batch, n_q, pool->n_kv, pool->d_head, max_blocks_per_seq,
                                               pool->partition_tokens);
    pkv_status st = ensure_workspace(pool, need);
    if (st != PKV_OK) return st;

    const int64_t P = (int64_t)batch * nps;
    uint8_t *ws = static_cast<uint8_t *>(pool->ws);
    DecodeArgs a;
    a.k_pool = static_cast<const uint8_t *>(pool->k);
    a.v_pool = static_cast<const uint8_t *>(pool->v);
    a.num_blocks = pool->num_blocks;
    a.n_kv = pool->n_kv;
    a.n_q = n_q;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.W = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.batch = batch;
    a.qscale = scale * kLog2e;
    a.scales = pool->scales;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.part_start = reinterpret_cast<int32_t *>(ws);
    a.ws_ml = reinterpret_cast<float2 *>(ws + align256(4 * (size_t)(batch + 1)));
    a.ws_o = reinterpret_cast<float *>(ws + align256(4 * (size_t)(batch + 1)) +
                                       align256(8 * (size_t)P * pool->n_kv * G));
    a.part_blocks = part_blocks;
    a.err = pool->err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pool->d_head == 128)
        return fp8 ? dispatch_g<128, true>(pool, a, G, nps, s) : dispatch_g<128, false>(pool, a, G, nps, s);
    return fp8 ? dispatch_g<64, true>(pool, a, G, nps, s) : dispatch_g<64, false>(pool, a, G, nps, s);
}
