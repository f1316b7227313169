// Block management on the device: copy-on-write copies and swapping blocks
// to and from host memory ("KV cache, PagedAttention and FlashAttention",
// Problem 4, "The idea": blocks shared by several sequences carry a
// reference count and are copied before a write; a preempted sequence's
// blocks can be swapped to CPU memory), plus the host-side refcounted block
// allocator that decides which blocks those are.
//
// A block of the pool is n_kv contiguous (block, KV head) entries of 16 key
// rows and 16 value rows (and for a 4-bit pool 16 value (scale, zero point)
// pairs).  A block's entry in a host swap buffer is [K bytes][V bytes][value
// parameters, 4-bit pools only]: the key rows of every head, then the value
// rows, then the parameters (block_bytes, block_bytes and param_bytes).  Every
// kernel here moves whole entries in 16-byte vectors, grid-stride over
// (block, 16-byte chunk of the entry): a pure copy, bound by HBM for device
// copies and by the CPU-GPU link for swaps.  Swaps read and write pinned host memory
// directly from the kernel (the host buffer is mapped into the device's
// address space), with no staging copy.
#include "pkv_internal.cuh"

#include <algorithm>
#include <map>
#include <mutex>
#include <set>
#include <vector>

namespace pkv {

struct BlockMoveArgs {
    uint8_t *pool;                 // the pool's first (block, KV head) entry
    const int32_t *src_ids, *dst_ids;  // block ids per pair (copy: both; swap-out: src; swap-in: dst)
    uint8_t *host;                 // swap buffer [n][entry bytes] (device address of pinned memory)
    int64_t n, num_blocks, block_bytes, param_bytes;  // image entry bytes = 2 block_bytes + param_bytes
    int64_t head_entry;            // bytes of a (block, KV head) entry in the pool
    int64_t head_rows;             // bytes of one head's 16 key (or value) rows: a power of two
    int rows_shift;                // log2(head_rows)
    int n_kv;
    unsigned *err;
};

// Byte `off` of a block's swap-image entry: where it sits in the pool is
// base + id * stride + off for block id.
struct EntryByte {
    uint8_t *base;
    int64_t stride, off;
};

__device__ __forceinline__ EntryByte entry_byte(const BlockMoveArgs &a, int64_t off)
{
    // the head's entry, and the section within it (16-byte chunks never straddle heads); section
    // sizes are powers of two, so the head is a shift
    int64_t sec = 0;
    int sh = a.rows_shift;
    if (off >= 2 * a.block_bytes) {  // 4-bit value parameters: 16 rows x 8 bytes per head
        off -= 2 * a.block_bytes;
        sec = 2 * a.head_rows;
        sh = 7;
    } else if (off >= a.block_bytes) {  // value rows
        off -= a.block_bytes;
        sec = a.head_rows;
    }
    const int64_t g = off >> sh;
    return {a.pool, a.n_kv * a.head_entry, g * a.head_entry + sec + (off & ((int64_t(1) << sh) - 1))};
}

enum MoveKind { kCopy = 0, kSwapOut = 1, kSwapIn = 2 };

template <int KIND>
__global__ void __launch_bounds__(256) block_move_kernel(BlockMoveArgs a)
{
    griddep_wait();  // ids and blocks may come from the previous kernel on the stream
    griddep_launch_dependents();
    const int64_t entry = 2 * a.block_bytes + a.param_bytes;
    const int64_t chunks = entry / 16;               // per block
    const int64_t total = a.n * chunks;              // (pair, chunk)
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t pair = i / chunks;
        const int64_t c = i - pair * chunks;
        // a copy moves the block's n_kv contiguous entries as they are; a swap maps each chunk of the
        // host image to its place in the entries
        const EntryByte e = KIND == kCopy ? EntryByte{a.pool, a.n_kv * a.head_entry, c * 16} : entry_byte(a, c * 16);
        if constexpr (KIND == kCopy) {
            const int64_t s = a.src_ids[pair], d = a.dst_ids[pair];
            if (s < 0 || s >= a.num_blocks || d < 0 || d >= a.num_blocks) {
                if (c == 0) atomicOr(a.err, PKV_DEVERR_BLOCK_RANGE);
                continue;
            }
            *reinterpret_cast<uint4 *>(e.base + d * e.stride + e.off) = ldg_nc_v4(e.base + s * e.stride + e.off);
        } else if constexpr (KIND == kSwapOut) {
            const int64_t s = a.src_ids[pair];
            if (s < 0 || s >= a.num_blocks) {
                if (c == 0) atomicOr(a.err, PKV_DEVERR_BLOCK_RANGE);
                continue;
            }
            *reinterpret_cast<uint4 *>(a.host + pair * entry + c * 16) = ldg_nc_v4(e.base + s * e.stride + e.off);
        } else {
            const int64_t d = a.dst_ids[pair];
            if (d < 0 || d >= a.num_blocks) {
                if (c == 0) atomicOr(a.err, PKV_DEVERR_BLOCK_RANGE);
                continue;
            }
            *reinterpret_cast<uint4 *>(e.base + d * e.stride + e.off) =
                *reinterpret_cast<const uint4 *>(a.host + pair * entry + c * 16);
        }
    }
}

template <int KIND>
static pkv_status launch_move(pkv_pool *pool, const BlockMoveArgs &a, cudaStream_t s, const char *what)
{
    const int64_t total = a.n * ((2 * a.block_bytes + a.param_bytes) / 16);
    int64_t blocks = (total + 255) / 256;
    blocks = std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)pool->num_sms * 8));
    LaunchScope ls(pool, kBlocks, s);
    cudaError_t e = launch_pdl(block_move_kernel<KIND>, dim3((unsigned)blocks), dim3(256), 0, s, a);
    ls.done();
    if (e != cudaSuccess) return cuda_fail(e, what);
    return PKV_OK;
}

static int64_t block_bytes_of(const pkv_pool *pool)
{
    return (int64_t)(pool->bytes_per_array / (size_t)pool->num_blocks);
}

// A 4-bit block's value parameters: (scale, zero point) fp32 per token row.
static int64_t param_bytes_of(const pkv_pool *pool)
{
    return pool->dtype == PKV_INT4 ? (int64_t)pool->n_kv * kBlockSize * 2 * (int64_t)sizeof(float) : 0;
}

static BlockMoveArgs move_args(pkv_pool *pool, int64_t n)
{
    BlockMoveArgs a = {};
    a.pool = static_cast<uint8_t *>(pool->k);
    a.n = n;
    a.num_blocks = pool->num_blocks;
    a.block_bytes = block_bytes_of(pool);
    a.param_bytes = param_bytes_of(pool);
    a.head_entry = kv_entry_bytes(pool->dtype, pool->d_head);
    a.head_rows = kv_v_offset(pool->dtype, pool->d_head);
    a.rows_shift = 0;
    while ((int64_t(1) << a.rows_shift) < a.head_rows) ++a.rows_shift;
    a.n_kv = pool->n_kv;
    a.err = pool->err;
    return a;
}

// Device address of a pinned host buffer, or null when `p` is not pinned
// host memory this device can reach.
}  // namespace pkv

using namespace pkv;

extern "C" int64_t kv_block_bytes(const pkv_pool *pool)
{
    return pool ? block_bytes_of(pool) : -1;
}

extern "C" int64_t kv_swap_entry_bytes(const pkv_pool *pool)
{
    return pool ? 2 * block_bytes_of(pool) + param_bytes_of(pool) : -1;
}

extern "C" pkv_status kv_block_copy(pkv_pool *pool, const int32_t *src_blocks, const int32_t *dst_blocks, int64_t n,
                                    void *stream)
{
    if (!pool) return fail(PKV_EINVAL, "kv_block_copy: NULL pool");
    if (n < 0) return fail(PKV_EINVAL, "kv_block_copy: n < 0");
    if (n == 0) return PKV_OK;
    if (!src_blocks || !dst_blocks) return fail(PKV_EINVAL, "kv_block_copy: NULL device pointer");
    if (((uintptr_t)src_blocks | (uintptr_t)dst_blocks) & 3u)
        return fail(PKV_EINVAL, "kv_block_copy: block id arrays must be 4-byte aligned");
    BlockMoveArgs a = move_args(pool, n);
    a.src_ids = src_blocks;
    a.dst_ids = dst_blocks;
    return launch_move<kCopy>(pool, a, static_cast<cudaStream_t>(stream), "kv_block_copy");
}

extern "C" pkv_status kv_swap_out(pkv_pool *pool, const int32_t *blocks, int64_t n, void *host_dst, void *stream)
{
    if (!pool) return fail(PKV_EINVAL, "kv_swap_out: NULL pool");
    if (n < 0) return fail(PKV_EINVAL, "kv_swap_out: n < 0");
    if (n == 0) return PKV_OK;
    if (!blocks || !host_dst) return fail(PKV_EINVAL, "kv_swap_out: NULL pointer");
    if (((uintptr_t)blocks & 3u) || ((uintptr_t)host_dst & 15u))
        return fail(PKV_EINVAL, "kv_swap_out: ids must be 4-byte and the host buffer 16-byte aligned");
    void *dev = mapped_host_ptr(host_dst);
    if (!dev) return fail(PKV_EINVAL, "kv_swap_out: host buffer is not pinned host memory (cudaHostAlloc / cudaHostRegister)");
    BlockMoveArgs a = move_args(pool, n);
    a.src_ids = blocks;
    a.host = static_cast<uint8_t *>(dev);
    return launch_move<kSwapOut>(pool, a, static_cast<cudaStream_t>(stream), "kv_swap_out");
}

extern "C" pkv_status kv_swap_in(pkv_pool *pool, const void *host_src, const int32_t *blocks, int64_t n, void *stream)
{
    if (!pool) return fail(PKV_EINVAL, "kv_swap_in: NULL pool");
    if (n < 0) return fail(PKV_EINVAL, "kv_swap_in: n < 0");
    if (n == 0) return PKV_OK;
    if (!blocks || !host_src) return fail(PKV_EINVAL, "kv_swap_in: NULL pointer");
    if (((uintptr_t)blocks & 3u) || ((uintptr_t)host_src & 15u))
        return fail(PKV_EINVAL, "kv_swap_in: ids must be 4-byte and the host buffer 16-byte aligned");
    void *dev = mapped_host_ptr(host_src);
    if (!dev) return fail(PKV_EINVAL, "kv_swap_in: host buffer is not pinned host memory (cudaHostAlloc / cudaHostRegister)");
    BlockMoveArgs a = move_args(pool, n);
    a.dst_ids = blocks;
    a.host = static_cast<uint8_t *>(dev);
    return launch_move<kSwapIn>(pool, a, static_cast<cudaStream_t>(stream), "kv_swap_in");
}

// ---------------------------------------------------------------------------
// Refcounted block allocator (host)
//
// The block manager the pages pair with the block table: physical blocks are
// handed out on demand, shared by reference count (parallel samples, beam
// branches, a common prompt prefix), and a shared block is replaced by a
// private copy before anyone writes into it.  Free blocks are handed out
// lowest id first, so a sequence of calls has one result.
// ---------------------------------------------------------------------------

struct pkv_alloc {
    std::mutex mu;
    std::vector<int32_t> ref;
    std::set<int32_t> free_ids;
};

extern "C" pkv_status kv_alloc_create(int64_t num_blocks, pkv_alloc **out)
{
    if (!out) return fail(PKV_EINVAL, "kv_alloc_create: NULL out");
    *out = nullptr;
    if (num_blocks <= 0 || num_blocks > INT32_MAX)
        return fail(PKV_EINVAL, "kv_alloc_create: num_blocks %lld out of range", (long long)num_blocks);
    pkv_alloc *a = new (std::nothrow) pkv_alloc;
    if (!a) return fail(PKV_ENOMEM, "kv_alloc_create: out of host memory");
    try {
        a->ref.assign((size_t)num_blocks, 0);
        for (int64_t i = 0; i < num_blocks; ++i) a->free_ids.insert(a->free_ids.end(), (int32_t)i);
    } catch (...) {
        delete a;
        return fail(PKV_ENOMEM, "kv_alloc_create: out of host memory");
    }
    *out = a;
    return PKV_OK;
}

extern "C" pkv_status kv_alloc_destroy(pkv_alloc *a)
{
    delete a;
    return PKV_OK;
}

extern "C" int64_t kv_alloc_free_blocks(pkv_alloc *a)
{
    if (!a) return -1;
    std::lock_guard<std::mutex> g(a->mu);
    return (int64_t)a->free_ids.size();
}

extern "C" pkv_status kv_alloc_refcount(pkv_alloc *a, int32_t id, int32_t *out)
{
    if (!a || !out) return fail(PKV_EINVAL, "kv_alloc_refcount: NULL argument");
    std::lock_guard<std::mutex> g(a->mu);
    if (id < 0 || (size_t)id >= a->ref.size()) return fail(PKV_ERANGE, "kv_alloc_refcount: block %d out of range", id);
    *out = a->ref[(size_t)id];
    return PKV_OK;
}

extern "C" pkv_status kv_alloc_take(pkv_alloc *a, int64_t n, int32_t *ids_out)
{
    if (!a) return fail(PKV_EINVAL, "kv_alloc_take: NULL allocator");
    if (n < 0) return fail(PKV_EINVAL, "kv_alloc_take: n < 0");
    if (n == 0) return PKV_OK;
    if (!ids_out) return fail(PKV_EINVAL, "kv_alloc_take: NULL ids_out");
    std::lock_guard<std::mutex> g(a->mu);
    if ((int64_t)a->free_ids.size() < n)
        return fail(PKV_ENOMEM, "kv_alloc_take: %lld blocks wanted, %zu free", (long long)n, a->free_ids.size());
    for (int64_t i = 0; i < n; ++i) {
        const int32_t id = *a->free_ids.begin();
        a->free_ids.erase(a->free_ids.begin());
        a->ref[(size_t)id] = 1;
        ids_out[i] = id;
    }
    return PKV_OK;
}

// Checks that every id is in range and held (refcount > 0), counting
// repeats: a block listed k times must hold at least k references when
// `need_refs` is set (releases), at least one otherwise (shares).
static pkv_status check_held(pkv_alloc *a, const int32_t *ids, int64_t n, bool need_refs, const char *what)
{
    std::vector<int32_t> seen;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        if (id < 0 || (size_t)id >= a->ref.size()) return fail(PKV_ERANGE, "%s: block %d out of range", what, id);
        if (a->ref[(size_t)id] <= 0) return fail(PKV_EINVAL, "%s: block %d is not allocated", what, id);
        if (need_refs) seen.push_back(id);
    }
    if (need_refs && n > 1) {
        std::sort(seen.begin(), seen.end());
        for (size_t i = 0; i < seen.size();) {
            size_t j = i;
            while (j < seen.size() && seen[j] == seen[i]) ++j;
            if ((int64_t)(j - i) > a->ref[(size_t)seen[i]])
                return fail(PKV_EINVAL, "%s: block %d released %zu times but holds %d references", what, seen[i],
                            j - i, a->ref[(size_t)seen[i]]);
            i = j;
        }
    }
    return PKV_OK;
}

extern "C" pkv_status kv_alloc_share(pkv_alloc *a, const int32_t *ids, int64_t n)
{
    if (!a) return fail(PKV_EINVAL, "kv_alloc_share: NULL allocator");
    if (n < 0) return fail(PKV_EINVAL, "kv_alloc_share: n < 0");
    if (n == 0) return PKV_OK;
    if (!ids) return fail(PKV_EINVAL, "kv_alloc_share: NULL ids");
    std::lock_guard<std::mutex> g(a->mu);
    pkv_status st = check_held(a, ids, n, false, "kv_alloc_share");
    if (st != PKV_OK) return st;
    for (int64_t i = 0; i < n; ++i) a->ref[(size_t)ids[i]] += 1;
    return PKV_OK;
}

extern "C" pkv_status kv_alloc_release(pkv_alloc *a, const int32_t *ids, int64_t n)
{
    if (!a) return fail(PKV_EINVAL, "kv_alloc_release: NULL allocator");
    if (n < 0) return fail(PKV_EINVAL, "kv_alloc_release: n < 0");
    if (n == 0) return PKV_OK;
    if (!ids) return fail(PKV_EINVAL, "kv_alloc_release: NULL ids");
    std::lock_guard<std::mutex> g(a->mu);
    pkv_status st = check_held(a, ids, n, true, "kv_alloc_release");
    if (st != PKV_OK) return st;
    for (int64_t i = 0; i < n; ++i)
        if (--a->ref[(size_t)ids[i]] == 0) a->free_ids.insert(ids[i]);
    return PKV_OK;
}

extern "C" pkv_status kv_alloc_prepare_write(pkv_alloc *a, int32_t *ids, int64_t n, int32_t *copy_src,
                                             int32_t *copy_dst, int64_t *n_copies)
{
    if (!a) return fail(PKV_EINVAL, "kv_alloc_prepare_write: NULL allocator");
    if (n < 0) return fail(PKV_EINVAL, "kv_alloc_prepare_write: n < 0");
    if (!n_copies) return fail(PKV_EINVAL, "kv_alloc_prepare_write: NULL n_copies");
    *n_copies = 0;
    if (n == 0) return PKV_OK;
    if (!ids || !copy_src || !copy_dst) return fail(PKV_EINVAL, "kv_alloc_prepare_write: NULL array");
    std::lock_guard<std::mutex> g(a->mu);
    pkv_status st = check_held(a, ids, n, false, "kv_alloc_prepare_write");
    if (st != PKV_OK) return st;
    // how many copies: walk the list as the update below will, on scratch counts
    std::map<int32_t, int32_t> ref_after;
    int64_t need = 0;
    for (int64_t i = 0; i < n; ++i) {
        auto it = ref_after.find(ids[i]);
        int32_t &r = it != ref_after.end() ? it->second : (ref_after[ids[i]] = a->ref[(size_t)ids[i]]);
        if (r > 1) {
            ++need;
            --r;
        }
    }
    if ((int64_t)a->free_ids.size() < need)
        return fail(PKV_ENOMEM, "kv_alloc_prepare_write: %lld copies needed, %zu blocks free", (long long)need,
                    a->free_ids.size());
    int64_t k = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        if (a->ref[(size_t)id] > 1) {
            const int32_t fresh = *a->free_ids.begin();
            a->free_ids.erase(a->free_ids.begin());
            a->ref[(size_t)fresh] = 1;
            a->ref[(size_t)id] -= 1;
            copy_src[k] = id;
            copy_dst[k] = fresh;
            ++k;
            ids[i] = fresh;
        }
    }
    *n_copies = k;
    return PKV_OK;
}
