// Append / scatter: write each token's new key and value rows into its slot
// of the block pool ("The KV Cache from First Principles", "Deriving the
// cache": k_t and v_t are computed once and appended; "KV cache,
// PagedAttention and FlashAttention", Problem 4: slot = physical block x B +
// offset).  FP8 pools quantise on the way in: E4M3(fp32(x) / scale[g]),
// round to nearest even, saturating.
//
// Work split: one group of D/8 lanes per (token, KV head) row, each lane
// moving 8 elements (one 16-byte load of bf16 per array).  Grid-stride over
// rows, so a per-step append (tens of rows) and a bulk prefill (millions)
// use the same kernel.  Memory-bound: per row it reads 2*D*2 bytes and
// writes 2*D*e bytes.
#include "pkv_internal.cuh"

#include <algorithm>

namespace pkv {

struct AppendArgs {
    uint8_t *k_pool;                      // the pool's first (block, KV head) entry
    int64_t num_blocks;
    int n_kv;
    const __nv_bfloat16 *k_new, *v_new;  // [T][n_kv][D]
    const int64_t *slot_mapping;          // [T]
    int64_t n_tokens;
    const float *scales;                  // [2*n_kv] (FP8 only)
    const float *k_params;                // 4-bit: [2][n_kv][D] key scales, then zero points
    // 4-bit step mode (when step_tables is set): token t is sequence t's newest
    // one, at position context_lens[t] - 1 of its dense table row
    const int32_t *step_tables, *step_lens;
    int step_W;
    unsigned *err;
};

template <int D, bool FP8>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a)
{
    constexpr int LPR = D / 8;  // lanes per row
    constexpr int E = FP8 ? 1 : 2;
    griddep_wait();  // inputs may come from the previous kernel on the stream
    griddep_launch_dependents();
    const int64_t rows = a.n_tokens * a.n_kv;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int sub = (int)(gid % LPR);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x / LPR;
    const int64_t slots = a.num_blocks * kBlockSize;
    for (int64_t row = gid / LPR; row < rows; row += stride) {
        const int64_t t = row / a.n_kv;
        const int g = (int)(row - t * a.n_kv);
        const int64_t slot = a.slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= slots) {
            if (sub == 0) atomicOr(a.err, PKV_DEVERR_SLOT_RANGE);
            continue;
        }
        const int64_t blk = slot / kBlockSize;
        const int64_t off = slot - blk * kBlockSize;
        // key row `off` of the (block, KV head) entry; its value row 16 rows further
        const int64_t dst = ((blk * a.n_kv + g) * 2 * kBlockSize + off) * (D * E) + sub * 8 * E;
        const int64_t vdst = dst + kBlockSize * D * E;
        const int64_t src = (t * a.n_kv + g) * D + sub * 8;
        const uint4 kr = ldg_nc_v4(a.k_new + src);
        const uint4 vr = ldg_nc_v4(a.v_new + src);
        if constexpr (!FP8) {
            *reinterpret_cast<uint4 *>(a.k_pool + dst) = kr;
            *reinterpret_cast<uint4 *>(a.k_pool + vdst) = vr;
        } else {
            const float ks = a.scales[g];
            const float vs = a.scales[a.n_kv + g];
            const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
            const uint32_t vw[4] = {vr.x, vr.y, vr.z, vr.w};
            uint32_t ko[2], vo[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 kf = bf16x2_to_f32x2(kw[i]);
                const float2 vf = bf16x2_to_f32x2(vw[i]);
                // correctly rounded fp32 division, then RN + satfinite to E4M3
                const uint32_t kq = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(kf.x, ks), __fdiv_rn(kf.y, ks)), __NV_SATFINITE, __NV_E4M3);
                const uint32_t vq = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(vf.x, vs), __fdiv_rn(vf.y, vs)), __NV_SATFINITE, __NV_E4M3);
                if (i & 1) {
                    ko[i >> 1] |= kq << 16;
                    vo[i >> 1] |= vq << 16;
                } else {
                    ko[i >> 1] = kq;
                    vo[i >> 1] = vq;
                }
            }
            *reinterpret_cast<uint2 *>(a.k_pool + dst) = make_uint2(ko[0], ko[1]);
            *reinterpret_cast<uint2 *>(a.k_pool + vdst) = make_uint2(vo[0], vo[1]);
        }
    }
}

// 4-bit code of x: clamp(rint((x - z) / s), 0, 15), each step correctly
// rounded in fp32 (round half to even), NaN to 0.
__device__ __forceinline__ uint32_t int4_code(float x, float s, float z)
{
    const float r = rintf(__fdiv_rn(__fsub_rn(x, z), s));
    return r >= 0.0f ? (uint32_t)fminf(r, 15.0f) : 0u;
}

// 4-bit pools: keys take their channel's (scale, zero point) from the pool;
// each value row gets scale (max - min) / 15 (1 if the row is constant) and
// zero point min + 0 (no negative zero), found by reducing min and max over
// the D/8 lanes of the row.  Eight codes per lane, packed two per byte with
// the even channel in the low nibble: one 32-bit store per lane and array,
// into the (block, KV head) entry (key codes, value codes, value parameters).
template <int D>
__global__ void __launch_bounds__(256) append_int4_kernel(AppendArgs a)
{
    constexpr int LPR = D / 8;  // lanes per row (8 or 16): a row never straddles a warp
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const unsigned group = ((1u << LPR) - 1u) << (lane & ~(LPR - 1));
    const int64_t rows = a.n_tokens * a.n_kv;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int sub = (int)(gid % LPR);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x / LPR;
    const int64_t slots = a.num_blocks * kBlockSize;
    for (int64_t row = gid / LPR; row < rows; row += stride) {
        const int64_t t = row / a.n_kv;
        const int g = (int)(row - t * a.n_kv);
        int64_t slot;
        if (a.step_tables) {  // the slot of position C-1 through the table (C = 0: nothing to append)
            const int c = a.step_lens[t];
            if (c <= 0) continue;
            const int j = (c - 1) / kBlockSize;
            if (j >= a.step_W) {
                if (sub == 0) atomicOr(a.err, PKV_DEVERR_CTX_RANGE);
                continue;
            }
            const int32_t phys = a.step_tables[t * a.step_W + j];
            slot = phys < 0 ? -1 : (int64_t)phys * kBlockSize + (c - 1) % kBlockSize;
        } else {
            slot = a.slot_mapping[t];
        }
        if (slot < 0) continue;  // the row's lanes agree: same slot
        if (slot >= slots) {
            if (sub == 0) atomicOr(a.err, PKV_DEVERR_SLOT_RANGE);
            continue;
        }
        const int64_t blk = slot / kBlockSize;
        const int off = (int)(slot - blk * kBlockSize);  // row in the block
        uint8_t *entry = a.k_pool + (blk * a.n_kv + g) * i4_entry_bytes(D);
        const int64_t src = (t * a.n_kv + g) * D + sub * 8;
        const uint4 kr = ldg_nc_v4(a.k_new + src);
        const uint4 vr = ldg_nc_v4(a.v_new + src);
        const uint32_t kw4[4] = {kr.x, kr.y, kr.z, kr.w}, vw4[4] = {vr.x, vr.y, vr.z, vr.w};
        float kf[8], vf[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 k2 = bf16x2_to_f32x2(kw4[i]), v2 = bf16x2_to_f32x2(vw4[i]);
            kf[2 * i] = k2.x;
            kf[2 * i + 1] = k2.y;
            vf[2 * i] = v2.x;
            vf[2 * i + 1] = v2.y;
        }
        const float *ks = a.k_params + (int64_t)g * D + sub * 8;
        const float *kz = a.k_params + (int64_t)(a.n_kv + g) * D + sub * 8;
        uint32_t kc = 0, vc = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) kc |= int4_code(kf[i], ks[i], kz[i]) << (4 * i);
        float mn = vf[0], mx = vf[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            mn = fminf(mn, vf[i]);
            mx = fmaxf(mx, vf[i]);
        }
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(group, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(group, mx, o));
        }
        float sc = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
        if (sc == 0.0f) sc = 1.0f;
        const float z = __fadd_rn(mn, 0.0f);
#pragma unroll
        for (int i = 0; i < 8; ++i) vc |= int4_code(vf[i], sc, z) << (4 * i);
        *reinterpret_cast<uint32_t *>(entry + off * (D / 2) + sub * 4) = kc;
        *reinterpret_cast<uint32_t *>(entry + i4_v_offset(D) + off * (D / 2) + sub * 4) = vc;
        if (sub == 0) *reinterpret_cast<float2 *>(entry + i4_params_offset(D) + off * 8) = make_float2(sc, z);
    }
}

template <int D>
static cudaError_t launch_append_int4(const AppendArgs &a, int num_sms, cudaStream_t s)
{
    constexpr int LPR = D / 8;
    constexpr int kThreads = 256;
    const int64_t lanes = a.n_tokens * a.n_kv * LPR;
    int64_t blocks = (lanes + kThreads - 1) / kThreads;
    blocks = std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)num_sms * 8));
    return launch_pdl(append_int4_kernel<D>, dim3((unsigned)blocks), dim3(kThreads), 0, s, a);
}

template <int D, bool FP8>
static cudaError_t launch_append(const AppendArgs &a, int num_sms, cudaStream_t s)
{
    constexpr int LPR = D / 8;
    constexpr int kThreads = 256;
    const int64_t lanes = a.n_tokens * a.n_kv * LPR;
    int64_t blocks = (lanes + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(append_kernel<D, FP8>, dim3((unsigned)blocks), dim3(kThreads), 0, s, a);
}

pkv_status probe_kernels()
{
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, append_kernel<128, false>);
    if (e != cudaSuccess)
        return fail(e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ? PKV_ECUDA : PKV_EUNSUPPORTED,
                    "this library runs on sm_103 (GB300) only: %s", cudaGetErrorString(e));
    return PKV_OK;
}

}  // namespace pkv

namespace pkv {

// The append half of a 4-bit pool's decode step: each sequence's newest
// token (k_new, v_new [batch][n_kv][d_head]) into the slot of position
// context_lens[b] - 1 through its dense table row.
pkv_status append_step_int4(pkv_pool *pool, const void *k_new, const void *v_new, const int32_t *tables, int W,
                            const int32_t *lens, int batch, cudaStream_t s)
{
    AppendArgs a;
    a.k_pool = static_cast<uint8_t *>(pool->k);
    a.num_blocks = pool->num_blocks;
    a.n_kv = pool->n_kv;
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.slot_mapping = nullptr;
    a.n_tokens = batch;
    a.scales = pool->scales;
    a.k_params = pool->k_params;
    a.step_tables = tables;
    a.step_lens = lens;
    a.step_W = W;
    a.err = pool->err;
    LaunchScope ls(pool, kAppend, s);
    cudaError_t e = pool->d_head == 128 ? launch_append_int4<128>(a, pool->num_sms, s)
                                        : launch_append_int4<64>(a, pool->num_sms, s);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, "append (4-bit step) launch");
    return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_kv_append(pkv_pool *pool, const void *k_new, const void *v_new,
                                      const int64_t *slot_mapping, int64_t n_tokens, void *stream)
{
    if (!pool) return fail(PKV_EINVAL, "paged_kv_append: NULL pool");
    if (n_tokens < 0) return fail(PKV_EINVAL, "paged_kv_append: n_tokens < 0");
    if (n_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping)
        return fail(PKV_EINVAL, "paged_kv_append: NULL device pointer");
    if (((uintptr_t)k_new | (uintptr_t)v_new) & 15u)
        return fail(PKV_EINVAL, "paged_kv_append: k_new/v_new must be 16-byte aligned");
    if ((uintptr_t)slot_mapping & 7u)
        return fail(PKV_EINVAL, "paged_kv_append: slot_mapping must be 8-byte aligned");
    const bool fp8 = pool->dtype == PKV_FP8_E4M3, i4 = pool->dtype == PKV_INT4;
    if (fp8 && !pool->scales_set)
        return fail(PKV_EINVAL, "paged_kv_append: FP8 pool needs kv_pool_set_fp8_scales first");
    if (i4 && !pool->scales_set)
        return fail(PKV_EINVAL, "paged_kv_append: 4-bit pool needs kv_pool_set_int4_key_params first");
    AppendArgs a;
    a.k_pool = static_cast<uint8_t *>(pool->k);
    a.num_blocks = pool->num_blocks;
    a.n_kv = pool->n_kv;
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.slot_mapping = slot_mapping;
    a.n_tokens = n_tokens;
    a.scales = pool->scales;
    a.k_params = pool->k_params;
    a.step_tables = a.step_lens = nullptr;
    a.step_W = 0;
    a.err = pool->err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    LaunchScope ls(pool, kAppend, s);
    cudaError_t e;
    if (i4)
        e = pool->d_head == 128 ? launch_append_int4<128>(a, pool->num_sms, s)
                                : launch_append_int4<64>(a, pool->num_sms, s);
    else if (pool->d_head == 128)
        e = fp8 ? launch_append<128, true>(a, pool->num_sms, s) : launch_append<128, false>(a, pool->num_sms, s);
    else
        e = fp8 ? launch_append<64, true>(a, pool->num_sms, s) : launch_append<64, false>(a, pool->num_sms, s);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, "paged_kv_append launch");
    return PKV_OK;
}
