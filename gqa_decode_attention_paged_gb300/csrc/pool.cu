// Pool lifetime, layout, FP8 scales, workspace, error word, timing and the
// host-only entry points of the C ABI (include/pagedkv.h).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>

#include <cudaTypedefs.h>

#include "pkv_internal.cuh"

namespace pkv {

static thread_local char g_msg[512] = "";

pkv_status fail(pkv_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

pkv_status cuda_fail(cudaError_t e, const char *what)
{
    snprintf(g_msg, sizeof g_msg, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
    if (e == cudaErrorMemoryAllocation) return PKV_ENOMEM;
    return PKV_ECUDA;
}

LaunchScope::LaunchScope(pkv_pool *p, int k, cudaStream_t s) : pool(p), kind(k), stream(s)
{
    std::lock_guard<std::mutex> g(pool->mu);
    pool->launches[kind] += 1;
    if (!pool->timing) return;
    for (cudaEvent_t *ev : {&a, &b}) {
        if (!pool->free_events.empty()) {
            *ev = pool->free_events.back();
            pool->free_events.pop_back();
        } else if (cudaEventCreate(ev) != cudaSuccess) {
            *ev = nullptr;
        }
    }
    if (a && b) cudaEventRecord(a, stream);
}

void LaunchScope::done()
{
    if (!a || !b) return;
    cudaEventRecord(b, stream);
    std::lock_guard<std::mutex> g(pool->mu);
    pool->pending.push_back(EventPair{a, b, kind});
}

pkv_status ensure_workspace(pkv_pool *pool, size_t bytes)
{
    if (bytes <= pool->ws_bytes) return PKV_OK;
    size_t want = bytes + bytes / 4;  // grow with headroom
    want = (want + (1u << 20) - 1) & ~size_t((1u << 20) - 1);
    if (pool->ws) {
        cudaError_t e = cudaFree(pool->ws);  // synchronises: no kernel still uses it
        pool->ws = nullptr;
        pool->ws_bytes = 0;
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
    }
    cudaError_t e = cudaMalloc(&pool->ws, want);
    if (e != cudaSuccess) {
        pool->ws = nullptr;
        return cuda_fail(e, "cudaMalloc(workspace)");
    }
    pool->ws_bytes = want;
    return PKV_OK;
}

pkv_status ensure_staging(pkv_pool *pool, size_t bytes)
{
    if (bytes <= pool->stage_bytes) return PKV_OK;
    if (pool->stage) {
        cudaError_t e = cudaFree(pool->stage);
        pool->stage = nullptr;
        pool->stage_bytes = 0;
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(staging)");
    }
    cudaError_t e = cudaMalloc(&pool->stage, bytes);
    if (e != cudaSuccess) {
        pool->stage = nullptr;
        return cuda_fail(e, "cudaMalloc(staging)");
    }
    pool->stage_bytes = bytes;
    return PKV_OK;
}

// The K and V arrays as 2-D tensors [blocks * n_kv * block_size rows][d_head]
// for tiled TMA: one box = 16 token rows of one (block, KV head) tile and up
// to 128 bytes of each row, with the matching shared-memory swizzle so that
// warp-wide fragment loads hit distinct banks.
static pkv_status tiled_encoder(PFN_cuTensorMapEncodeTiled_v12000 *out)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    static cudaError_t get_err = cudaSuccess;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        get_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void **>(&encode),
                                                   12000, cudaEnableDefault, &q);
        if (get_err == cudaSuccess && q != cudaDriverEntryPointSuccess) get_err = cudaErrorNotSupported;
    });
    if (get_err != cudaSuccess || !encode) return cuda_fail(get_err, "cuTensorMapEncodeTiled entry point");
    *out = encode;
    return PKV_OK;
}

void *mapped_host_ptr(const void *p)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
    return at.devicePointer;
}

pkv_status make_q_map(CUtensorMap *map, const void *q, int64_t n_rows, int n_q, int d_head, int heads, int tokens)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    pkv_status st = tiled_encoder(&encode);
    if (st != PKV_OK) return st;
    cuuint64_t dims[3] = {(cuuint64_t)d_head, (cuuint64_t)n_q, (cuuint64_t)n_rows};
    cuuint64_t strides[2] = {(cuuint64_t)d_head * 2, (cuuint64_t)n_q * d_head * 2};
    cuuint32_t box[3] = {(cuuint32_t)(d_head < 64 ? d_head : 64), (cuuint32_t)heads, (cuuint32_t)tokens};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled (queries) failed (%d)", (int)r);
    return PKV_OK;
}

pkv_status make_tensor_maps(pkv_pool *pool)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    pkv_status st = tiled_encoder(&encode);
    if (st != PKV_OK) return st;
    // the entries' rows: d_head bf16 or d_head E4M3 bytes each, 32 per entry (16 key rows, then 16
    // value rows); 16-row boxes (tm_block) and 32-row boxes (tm_entry) over the same rows
    const int elem = pool->dtype == PKV_BF16 ? 2 : 1;
    const uint64_t row_elems = (uint64_t)pool->d_head;
    const uint64_t row_bytes = row_elems * elem;
    const uint64_t rows = (uint64_t)pool->num_blocks * pool->n_kv * 2 * pool->block_size;
    if (rows >= (1ull << 31)) return fail(PKV_EUNSUPPORTED, "kv_pool_create: more than 2^31 key and value rows");
    const uint32_t box_bytes = row_bytes > 128 ? 128 : (uint32_t)row_bytes;
    cuuint64_t dims[2] = {(cuuint64_t)row_elems, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle sw = box_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                    : CU_TENSOR_MAP_SWIZZLE_32B;
    for (int which = 0; which < 2; ++which) {
        cuuint32_t box[2] = {box_bytes / (uint32_t)elem, (cuuint32_t)((which ? 2 : 1) * pool->block_size)};
        CUresult r = encode(which ? &pool->tm_entry : &pool->tm_block, dt, 2, pool->k, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    return PKV_OK;
}

// One warp waits on an mbarrier that nothing ever arrives at, with the same
// bounded wait the decode kernel uses; when the limit runs out it records
// PKV_DEVERR_TIMEOUT and returns.
__global__ void wait_selftest_kernel(unsigned *err, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
    if (__any_sync(0xffffffffu, !ok) && threadIdx.x == 0) atomicOr(err, PKV_DEVERR_TIMEOUT);
}

// Defined in append.cu / decode.cu: confirm the device can run our kernels.
pkv_status probe_kernels();
pkv_status decode_workspace_bytes(pkv_pool *pool, int batch, int n_q, int max_blocks_per_seq, size_t *bytes);

}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_string(pkv_status s)
{
    switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_EINVAL: return "PKV_EINVAL";
    case PKV_ERANGE: return "PKV_ERANGE";
    case PKV_ENOMEM: return "PKV_ENOMEM";
    case PKV_ECUDA: return "PKV_ECUDA";
    case PKV_EUNSUPPORTED: return "PKV_EUNSUPPORTED";
    case PKV_EDEVICE: return "PKV_EDEVICE";
    }
    return "PKV_UNKNOWN";
}

const char *pkv_last_error_message(void) { return g_msg; }

double kv_bytes_per_token(int32_t layers, int32_t n_kv, int32_t d_head, double bytes_per_value)
{
    if (layers < 0 || n_kv < 0 || d_head < 0 || !(bytes_per_value >= 0.0)) return -1.0;
    // keys and values (2) x layers x KV heads x head dim x bytes per value
    return 2.0 * (double)layers * (double)n_kv * (double)d_head * bytes_per_value;
}

pkv_status kv_pool_create(int64_t num_blocks, int32_t block_size, int32_t n_kv, int32_t d_head,
                          int32_t dtype, pkv_pool **out)
{
    g_msg[0] = '\0';
    if (!out) return fail(PKV_EINVAL, "kv_pool_create: out is NULL");
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0 || n_kv <= 0 || d_head <= 0)
        return fail(PKV_EINVAL, "kv_pool_create: sizes must be positive");
    if (block_size != kBlockSize)
        return fail(PKV_EUNSUPPORTED, "kv_pool_create: block_size %d unsupported (16 only)", block_size);
    if (d_head != 64 && d_head != 128)
        return fail(PKV_EUNSUPPORTED, "kv_pool_create: d_head %d unsupported (64 or 128)", d_head);
    if (n_kv > 256) return fail(PKV_EUNSUPPORTED, "kv_pool_create: n_kv %d > 256", n_kv);
    if (dtype != PKV_BF16 && dtype != PKV_FP8_E4M3 && dtype != PKV_INT4)
        return fail(PKV_EINVAL, "kv_pool_create: unknown dtype %d", dtype);
    const size_t row_bytes = dtype == PKV_BF16 ? 2 * (size_t)d_head : dtype == PKV_FP8_E4M3 ? d_head : d_head / 2;
    const size_t per_block = (size_t)n_kv * block_size * row_bytes;
    if ((size_t)num_blocks > ((size_t)1 << 46) / per_block)
        return fail(PKV_ERANGE, "kv_pool_create: pool too large");

    pkv_status st = probe_kernels();
    if (st != PKV_OK) return st;

    pkv_pool *p = new (std::nothrow) pkv_pool();
    if (!p) return fail(PKV_ENOMEM, "kv_pool_create: host allocation failed");
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "kv_pool_create: device query");
    }
    // paged_decode_attention_noalloc's scratch: its address is looked up now, which
    // (lazy module loading) also takes the array's memory now, before the pool's
    st = noalloc_scratch_address(&p->noalloc_scratch);
    if (st != PKV_OK) {
        delete p;
        return st;
    }
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->n_kv = n_kv;
    p->d_head = d_head;
    p->dtype = dtype;
    p->bytes_per_array = per_block * (size_t)num_blocks;
    // one allocation of (block, KV head) entries: key rows, value rows (and 4-bit value parameters)
    p->alloc_bytes = (size_t)num_blocks * n_kv * (size_t)kv_entry_bytes(dtype, d_head);
    const char *what = "cudaMalloc(pool)";
    e = cudaMalloc(&p->k, p->alloc_bytes);
    if (e == cudaSuccess) {
        p->v = static_cast<uint8_t *>(p->k) + kv_v_offset(dtype, d_head);
        if (dtype == PKV_INT4)
            p->v_params = reinterpret_cast<float *>(static_cast<uint8_t *>(p->k) + i4_params_offset(d_head));
    }
    if (e == cudaSuccess) { what = "cudaMalloc(scales)"; e = cudaMalloc(&p->scales, sizeof(float) * 2 * n_kv); }
    if (e == cudaSuccess) { what = "cudaMalloc(error word)"; e = cudaMalloc(&p->err, sizeof(unsigned)); }
    if (e == cudaSuccess && dtype == PKV_INT4) {
        what = "cudaMalloc(key params)";
        e = cudaMalloc(&p->k_params, sizeof(float) * 2 * n_kv * d_head);
        if (e == cudaSuccess) e = cudaMemset(p->k_params, 0, sizeof(float) * 2 * n_kv * d_head);
    }
    if (e == cudaSuccess) { what = "cudaMemset"; e = cudaMemset(p->k, 0, p->alloc_bytes); }
    if (e == cudaSuccess) e = cudaMemset(p->scales, 0, sizeof(float) * 2 * n_kv);
    if (e == cudaSuccess) e = cudaMemset(p->err, 0, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        pkv_status s = cuda_fail(e, what);
        kv_pool_destroy(p);
        return s;
    }
    st = dtype == PKV_INT4 ? PKV_OK : make_tensor_maps(p);
    if (st != PKV_OK) {
        kv_pool_destroy(p);
        return st;
    }
    *out = p;
    return PKV_OK;
}

pkv_status kv_pool_destroy(pkv_pool *pool)
{
    if (!pool) return PKV_OK;
    cudaDeviceSynchronize();
    cudaFree(pool->k);  // v (and v_params) point into the same allocation
    cudaFree(pool->scales);
    cudaFree(pool->k_params);
    cudaFree(pool->err);
    cudaFree(pool->ws);
    cudaFree(pool->stage);
    if (pool->host_graph) cudaGraphExecDestroy(pool->host_graph);
    if (pool->capture_stream) cudaStreamDestroy(pool->capture_stream);
    for (auto &pe : pool->pending) {
        cudaEventDestroy(pe.start);
        cudaEventDestroy(pe.stop);
    }
    for (cudaEvent_t ev : pool->free_events) cudaEventDestroy(ev);
    delete pool;
    return PKV_OK;
}

pkv_status kv_pool_set_fp8_scales(pkv_pool *pool, const float *k_scale_host, const float *v_scale_host)
{
    if (!pool || !k_scale_host || !v_scale_host)
        return fail(PKV_EINVAL, "kv_pool_set_fp8_scales: NULL argument");
    if (pool->dtype != PKV_FP8_E4M3)
        return fail(PKV_EINVAL, "kv_pool_set_fp8_scales: pool is not FP8");
    std::vector<float> s(2 * pool->n_kv);
    for (int g = 0; g < pool->n_kv; ++g) {
        s[g] = k_scale_host[g];
        s[pool->n_kv + g] = v_scale_host[g];
    }
    for (float x : s)
        if (!(x > 0.0f) || !isfinite(x))
            return fail(PKV_EINVAL, "kv_pool_set_fp8_scales: scales must be finite and > 0");
    cudaError_t e = cudaMemcpy(pool->scales, s.data(), sizeof(float) * s.size(), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "kv_pool_set_fp8_scales");
    pool->scales_set = true;
    return PKV_OK;
}

pkv_status kv_pool_set_int4_key_params(pkv_pool *pool, const float *k_scale_host, const float *k_zero_host)
{
    if (!pool || !k_scale_host || !k_zero_host) return fail(PKV_EINVAL, "kv_pool_set_int4_key_params: NULL argument");
    if (pool->dtype != PKV_INT4) return fail(PKV_EINVAL, "kv_pool_set_int4_key_params: pool is not 4-bit");
    const size_t n = (size_t)pool->n_kv * pool->d_head;
    std::vector<float> s(2 * n);
    for (size_t i = 0; i < n; ++i) {
        s[i] = k_scale_host[i];
        s[n + i] = k_zero_host[i];
        if (!(s[i] > 0.0f) || !isfinite(s[i]) || !isfinite(s[n + i]))
            return fail(PKV_EINVAL, "kv_pool_set_int4_key_params: scales must be finite and > 0, zeros finite");
    }
    cudaError_t e = cudaMemcpy(pool->k_params, s.data(), sizeof(float) * s.size(), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "kv_pool_set_int4_key_params");
    pool->scales_set = true;
    return PKV_OK;
}

pkv_status kv_pool_layout(const pkv_pool *pool, pkv_layout *out)
{
    if (!pool || !out) return fail(PKV_EINVAL, "kv_pool_layout: NULL argument");
    out->k = pool->k;
    out->v = pool->v;
    out->v_params = pool->v_params;
    out->v_params_bytes = pool->v_params ? (int64_t)pool->num_blocks * pool->n_kv * pool->block_size * 8 : 0;
    // strides in elements (bytes for 4-bit pools): an entry is 2 x 16 rows (+ 4-bit parameters)
    const int64_t elem = pool->dtype == PKV_BF16 ? 2 : 1;
    out->stride_token = pool->dtype == PKV_INT4 ? pool->d_head / 2 : pool->d_head;
    out->stride_head = kv_entry_bytes(pool->dtype, pool->d_head) / elem;
    out->stride_block = (int64_t)pool->n_kv * out->stride_head;
    out->alloc_bytes = (int64_t)pool->alloc_bytes;
    out->num_blocks = pool->num_blocks;
    out->block_size = pool->block_size;
    out->n_kv = pool->n_kv;
    out->d_head = pool->d_head;
    out->dtype = pool->dtype;
    out->bytes_per_array = (int64_t)pool->bytes_per_array;
    return PKV_OK;
}

pkv_status kv_pool_set_partition_tokens(pkv_pool *pool, int32_t tokens)
{
    if (!pool) return fail(PKV_EINVAL, "kv_pool_set_partition_tokens: NULL pool");
    if (tokens != 0 && (tokens < 16 || tokens > (1 << 20) || tokens % 16))
        return fail(PKV_ERANGE, "kv_pool_set_partition_tokens: %d is neither 0 nor a multiple of 16 in [16, 2^20]",
                    tokens);
    pool->partition_tokens = tokens;
    return PKV_OK;
}

pkv_status kv_pool_set_cascade_mode(pkv_pool *pool, int32_t mode)
{
    if (!pool) return fail(PKV_EINVAL, "kv_pool_set_cascade_mode: NULL pool");
    if (mode != PKV_CASCADE_AUTO && mode != PKV_CASCADE_ALWAYS && mode != PKV_CASCADE_NEVER)
        return fail(PKV_EINVAL, "kv_pool_set_cascade_mode: unknown mode %d", mode);
    pool->cascade_mode = mode;
    return PKV_OK;
}

pkv_status kv_pool_reserve_workspace(pkv_pool *pool, int32_t batch, int32_t n_q, int32_t max_blocks_per_seq)
{
    if (!pool || batch < 0 || n_q <= 0 || max_blocks_per_seq <= 0 || n_q % pool->n_kv)
        return fail(PKV_EINVAL, "kv_pool_reserve_workspace: bad argument");
    size_t bytes = 0;
    pkv_status st = decode_workspace_bytes(pool, batch, n_q, max_blocks_per_seq, &bytes);
    if (st != PKV_OK) return st;
    return ensure_workspace(pool, bytes);
}

pkv_status pkv_get_error(pkv_pool *pool, int32_t clear, uint32_t *bits)
{
    if (!pool) return fail(PKV_EINVAL, "pkv_get_error: NULL pool");
    unsigned v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, pool->err, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear) e = cudaMemset(pool->err, 0, sizeof(unsigned));
    if (e == cudaSuccess && clear) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "pkv_get_error");
    if (bits) *bits = v;
    if (v) return fail(PKV_EDEVICE, "device error bits 0x%x", v);
    return PKV_OK;
}

pkv_status pkv_selftest_wait_timeout(pkv_pool *pool, uint64_t limit_ns, void *stream)
{
    if (!pool) return fail(PKV_EINVAL, "pkv_selftest_wait_timeout: NULL pool");
    if (limit_ns < 1000 || limit_ns > kWaitLimitNs)
        return fail(PKV_ERANGE, "pkv_selftest_wait_timeout: limit must be in [1 us, 2 s]");
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(pool->err, limit_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "pkv_selftest_wait_timeout launch");
    return PKV_OK;
}

pkv_status pkv_timing_enable(pkv_pool *pool, int32_t on)
{
    if (!pool) return fail(PKV_EINVAL, "pkv_timing_enable: NULL pool");
    std::lock_guard<std::mutex> g(pool->mu);
    pool->timing = on != 0;
    return PKV_OK;
}

pkv_status pkv_timing_read(pkv_pool *pool, int32_t reset, pkv_timing *out)
{
    if (!pool) return fail(PKV_EINVAL, "pkv_timing_read: NULL pool");
    std::vector<EventPair> pend;
    {
        std::lock_guard<std::mutex> g(pool->mu);
        pend.swap(pool->pending);
    }
    pkv_status st = PKV_OK;
    for (auto &pe : pend) {
        cudaError_t e = cudaEventSynchronize(pe.stop);
        float ms = 0.0f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, pe.start, pe.stop);
        if (e != cudaSuccess && st == PKV_OK) st = cuda_fail(e, "pkv_timing_read");
        std::lock_guard<std::mutex> g(pool->mu);
        if (e == cudaSuccess) {
            pool->ms[pe.kind] += ms;
            pool->timed[pe.kind] += 1;
        }
        pool->free_events.push_back(pe.start);
        pool->free_events.push_back(pe.stop);
    }
    std::lock_guard<std::mutex> g(pool->mu);
    if (out) {
        out->append_launches = pool->launches[kAppend];
        out->decode_launches = pool->launches[kDecode];
        out->merge_launches = pool->launches[kMerge];
        out->prefix_launches = pool->launches[kPrefix];
        out->block_launches = pool->launches[kBlocks];
        out->block_ms = pool->ms[kBlocks];
        out->timed_block = pool->timed[kBlocks];
        out->launches = out->append_launches + out->decode_launches + out->merge_launches + out->prefix_launches +
                        out->block_launches;
        out->prefix_ms = pool->ms[kPrefix];
        out->timed_prefix = pool->timed[kPrefix];
        out->append_ms = pool->ms[kAppend];
        out->decode_ms = pool->ms[kDecode];
        out->merge_ms = pool->ms[kMerge];
        out->workspace_bytes = (int64_t)pool->ws_bytes;
        out->timed_append = pool->timed[kAppend];
        out->timed_decode = pool->timed[kDecode];
        out->timed_merge = pool->timed[kMerge];
    }
    if (reset) {
        for (int k = 0; k < kNumKinds; ++k) {
            pool->launches[k] = 0;
            pool->timed[k] = 0;
            pool->ms[k] = 0.0;
        }
    }
    return st;
}

}  // extern "C"
