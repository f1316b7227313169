// Internal declarations shared by the library's translation units: the pool
// object, status helpers and the inline-PTX wrappers for mbarriers and bulk
// (TMA) copies used by the kernels.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

#include "pagedkv.h"

namespace pkv {

constexpr int kBlockSize = 16;               // token slots per block
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded mbarrier waits: 2 s
constexpr int kDefaultPartitionTokens = 0;  // 0: equal work per CTA

// Every pool keeps what one (block, KV head) needs in one contiguous entry:
// its 16 key rows, then its 16 value rows (d bf16, d E4M3 bytes, or d/2 bytes
// of packed 4-bit codes per row), and for 4-bit pools then its 16 value rows'
// fp32 (scale, zero point) pairs.  Entries are [num_blocks][n_kv] in one
// allocation; each is a multiple of 16 bytes, so the decode kernel fetches
// one with a single copy (one TMA box per 128-byte column, or one bulk copy).
constexpr int64_t kv_row_bytes(int dtype, int d_head)
{
    return dtype == PKV_BF16 ? 2 * (int64_t)d_head : dtype == PKV_FP8_E4M3 ? d_head : d_head / 2;
}
constexpr int64_t kv_v_offset(int dtype, int d_head) { return kBlockSize * kv_row_bytes(dtype, d_head); }
constexpr int64_t kv_entry_bytes(int dtype, int d_head)
{
    return 2 * kv_v_offset(dtype, d_head) + (dtype == PKV_INT4 ? kBlockSize * 8 : 0);
}
constexpr int64_t i4_entry_bytes(int d_head) { return kv_entry_bytes(PKV_INT4, d_head); }
constexpr int64_t i4_v_offset(int d_head) { return kv_v_offset(PKV_INT4, d_head); }       // value codes
constexpr int64_t i4_params_offset(int d_head) { return 2 * kv_v_offset(PKV_INT4, d_head); }  // value (scale, zero)

enum KernelKind { kAppend = 0, kDecode = 1, kMerge = 2, kPrefix = 3, kBlocks = 4, kNumKinds = 5 };

struct EventPair {
    cudaEvent_t start, stop;
    int kind;
};

}  // namespace pkv

// The arguments a paged_decode_step_host graph was captured with.
struct pkv_host_step_key {
    const void *ptr[6] = {};  // q, k_new, v_new, block_tables, context_lens, out (host)
    int n_q = 0, W = 0, batch = 0, partition_tokens = 0;
    uint32_t scale_bits = 0;
    const void *stage = nullptr, *ws = nullptr;
    size_t ws_bytes = 0;
    void *stream = nullptr;
    bool operator==(const pkv_host_step_key &o) const
    {
        for (int i = 0; i < 6; ++i)
            if (ptr[i] != o.ptr[i]) return false;
        return n_q == o.n_q && W == o.W && batch == o.batch && partition_tokens == o.partition_tokens &&
               scale_bits == o.scale_bits && stage == o.stage && ws == o.ws && ws_bytes == o.ws_bytes &&
               stream == o.stream;
    }
};

struct pkv_pool {
    int device = 0;
    int num_sms = 0;
    int64_t num_blocks = 0;
    int block_size = 0, n_kv = 0, d_head = 0, dtype = 0;
    // one allocation of [num_blocks][n_kv] entries (kv_entry_bytes); k, v (and for 4-bit pools
    // v_params) point at the first entry's key rows, value rows (and value parameters)
    void *k = nullptr, *v = nullptr;
    size_t bytes_per_array = 0;       // bytes of K (and of V) data in the pool
    size_t alloc_bytes = 0;           // bytes of the allocation k points into
    float *scales = nullptr;          // device [2 * n_kv]: k scales then v scales
    // 4-bit pools: each value row's (scale, zero point), inside the entries, and the keys'
    // per-channel parameters [2][n_kv][d_head] fp32 (scales, then zero points)
    float *v_params = nullptr;
    float *k_params = nullptr;
    // TMA descriptors of the entries viewed as 2-D [rows = blocks*n_kv*32][d_head] (an entry's
    // key rows at 32 u .. 32 u + 15, its value rows after them), boxes of min(row bytes, 128)
    // bytes, swizzled (128 B, or 64 B for 64-byte rows): tm_block 16 rows high (one block's keys
    // or values: prefill), tm_entry 32 rows high (an entry's keys and values together: decode).
    // bf16 and FP8 pools only (4-bit entries are fetched by bulk copies).
    CUtensorMap tm_block, tm_entry;
    bool scales_set = false;
    unsigned *err = nullptr;          // device sticky error word
    void *ws = nullptr;               // split-KV workspace (grow-only)
    size_t ws_bytes = 0;
    void *stage = nullptr;            // device staging for paged_decode_step_host (grow-only)
    size_t stage_bytes = 0;
    int partition_tokens = pkv::kDefaultPartitionTokens;
    int cascade_mode = PKV_CASCADE_AUTO;  // paged_decode_attention_prefix: cascade or plain decode
    // device address of paged_decode_attention_noalloc's scratch array in the
    // context the pool was created in (looked up by kv_pool_create)
    void *noalloc_scratch = nullptr;
    // paged_decode_step_host: the launches of a call with pinned buffers, captured as a CUDA
    // graph and replayed while the call's arguments and the pool's buffers stay the same
    cudaGraphExec_t host_graph = nullptr;
    pkv_host_step_key host_key;
    cudaStream_t capture_stream = nullptr;
    // timing / launch accounting
    std::mutex mu;
    bool timing = false;
    std::vector<pkv::EventPair> pending;
    std::vector<cudaEvent_t> free_events;
    int64_t launches[pkv::kNumKinds] = {0, 0, 0};
    int64_t timed[pkv::kNumKinds] = {0, 0, 0};
    double ms[pkv::kNumKinds] = {0, 0, 0};
};

namespace pkv {

// Records a failure message for pkv_last_error_message() and returns `s`.
pkv_status fail(pkv_status s, const char *fmt, ...);
pkv_status cuda_fail(cudaError_t e, const char *what);

// Brackets a kernel launch with a timing event pair when timing is on, and
// counts the launch.  Usage: LaunchScope ls(pool, kind, stream); launch...;
// ls.done();
struct LaunchScope {
    pkv_pool *pool;
    int kind;
    cudaStream_t stream;
    cudaEvent_t a = nullptr, b = nullptr;
    LaunchScope(pkv_pool *p, int k, cudaStream_t s);
    void done();
};

pkv_status ensure_workspace(pkv_pool *pool, size_t bytes);
// The device address of paged_decode_attention_noalloc's scratch array on the
// current device (cudaGetSymbolAddress; loads the decode code if it is not
// loaded yet, which reserves the array's memory).
pkv_status noalloc_scratch_address(void **out);
pkv_status append_step_int4(pkv_pool *pool, const void *k_new, const void *v_new, const int32_t *tables, int W,
                            const int32_t *lens, int batch, cudaStream_t s);
pkv_status ensure_staging(pkv_pool *pool, size_t bytes);
pkv_status make_tensor_maps(pkv_pool *pool);
// The device address of pinned host memory (cudaHostAlloc / cudaHostRegister,
// mapped into the device's address space), or null for any other pointer.
void *mapped_host_ptr(const void *p);
// A 3-D tiled TMA map over a query array [n_rows][n_q][d_head] bf16: box of
// min(d_head, 64) columns x `heads` heads x `tokens` rows, 128-byte swizzle.
pkv_status make_q_map(CUtensorMap *map, const void *q, int64_t n_rows, int n_q, int d_head, int heads, int tokens);

// The cascade's prefix stage on the tensor cores (the prefill kernel in
// partial mode): every query row of every KV head against the shared blocks,
// cut into n_chunks chunks of chunk_blocks; one (m, l, O) partial per chunk,
// sequence and KV head into the merge workspace.
void prefix_stage_chunks(pkv_pool *pool, int batch, int n_q, int n_prefix_blocks, int *chunk_blocks, int *n_chunks);
pkv_status launch_prefix_stage(pkv_pool *pool, const void *q, int batch, int n_q, const int32_t *prefix_blocks,
                               int n_prefix_blocks, int chunk_blocks, int n_chunks, float qscale, float2 *ws_ml,
                               float *ws_o, int64_t pre_base, cudaStream_t s);

constexpr int kMaxBatch = 8192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

// Argument checks shared by the entry points that take device block tables.
pkv_status check_step_args(const pkv_pool *pool, const char *who, int n_q, int max_blocks_per_seq, int batch,
                           float scale);

// ---------------------------------------------------------------------------
// Device helpers (inline PTX)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// One-dimensional bulk copy global -> shared (TMA engine), completing
// `bytes` of transaction count on `bar`.  dst and src 16-byte aligned, bytes a
// multiple of 16.  evict-first L2 policy: K/V tiles are streamed once.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Tiled 2-D TMA load of one box at element coordinates (x, y) of `map`
// (a __grid_constant__ kernel parameter) into shared memory.
__device__ __forceinline__ void tma_load_2d(void *dst_smem, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Tiled 3-D TMA load of one box at element coordinates (x, y, z).
__device__ __forceinline__ void tma_load_3d(void *dst_smem, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: wait until the previous grid on the stream
// has completed and its memory is visible (a no-op when the kernel was not
// launched as a dependent), and let the next grid start launching early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` on `s` as a programmatic dependent of the previous work on
// the stream: its CTAs may become resident while that work drains; each
// kernel calls griddep_wait() before touching global memory.
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// bf16 pair packed in a 32-bit word -> two fp32 (exact).
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t u)
{
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}


}  // namespace pkv
