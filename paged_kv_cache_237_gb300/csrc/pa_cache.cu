// Cache write (reshape_and_cache) and copy-on-write block copy for sm_103a.
//
// Both are byte movers: every element is copied bit for bit with 16-byte
// vector loads and stores, coalesced along head_dim.
//
// Cache write: "PagedAttention" (robocikowo.com), "Jak dziala" -- blocks are
// allocated on demand as a sequence grows, so each new token's K/V lands in
// the slot its sequence's block table assigns; "PagedAttention et
// RadixAttention : parlons de KV Cache" (aitalk.it), third step.
// Block copy: same robocikowo.com page, "Komponenty" -- shared blocks are
// reference-counted and duplicated lazily when a sharer modifies them; the
// aitalk.it page's fourth step copies a block only when a request diverges.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_internal.h"

namespace pa {

// One CTA per token; threads stride over the token's 16-byte vectors of all
// KV heads, for K and V.
__global__ void __launch_bounds__(128)
    reshape_and_cache_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                             uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                             const int64_t *__restrict__ slot_mapping, int num_kv_heads,
                             int row_vecs /* 16-byte vectors per head row */, int block_size,
                             long long num_slots, int32_t *status) {
    const int t = blockIdx.x;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0) flag_status(status, PA_STATUS_BAD_SLOT);
        return;
    }
    const long long blk = slot / block_size, off = slot % block_size;
    const int total = num_kv_heads * row_vecs;
    const long long src0 = (long long)t * total;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int h = i / row_vecs, c = i % row_vecs;
        const long long dst = ((blk * num_kv_heads + h) * block_size + off) * row_vecs + c;
        const uint4 kv = k[src0 + i];
        const uint4 vv = v[src0 + i];
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

// grid (num_pairs, 2): blockIdx.y selects the K or the V cache.  Before
// writing, the CTA checks its pair against every other pair: a dst that is
// duplicated or that another pair reads is a race, so the pair is skipped and
// flagged.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                       const int64_t *__restrict__ pairs, int num_pairs, long long block_vecs,
                       int num_blocks, int32_t *status) {
    const int pidx = blockIdx.x;
    const int64_t src = pairs[2 * pidx], dst = pairs[2 * pidx + 1];
    __shared__ int conflict;
    if (threadIdx.x == 0) conflict = 0;
    __syncthreads();
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_status(status, PA_STATUS_BAD_PAIR);
        return;
    }
    if (src == dst) return;
    uint4 *cache = blockIdx.y == 0 ? k_cache : v_cache;
    const uint4 *from = cache + src * block_vecs;
    uint4 *to = cache + dst * block_vecs;
    // The first kPre vectors of the block are loaded before the conflict scan,
    // so that the scan's round trip overlaps theirs.  Reading src early is
    // safe: a pair whose dst is our src is itself flagged and skipped, so
    // nothing writes src during this launch.
    constexpr int kPre = 8;
    uint4 pre[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
        const long long i = threadIdx.x + static_cast<long long>(u) * blockDim.x;
        if (i < block_vecs) pre[u] = from[i];
    }
    for (int j = threadIdx.x; j < num_pairs; j += blockDim.x) {
        if (j == pidx) continue;
        const int64_t s2 = pairs[2 * j], d2 = pairs[2 * j + 1];
        if (d2 == dst || s2 == dst) conflict = 1;
    }
    __syncthreads();
    if (conflict) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_status(status, PA_STATUS_BAD_PAIR);
        return;
    }
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
        const long long i = threadIdx.x + static_cast<long long>(u) * blockDim.x;
        if (i < block_vecs) to[i] = pre[u];
    }
    long long i = threadIdx.x + static_cast<long long>(kPre) * blockDim.x;
    // four independent 16-byte loads in flight per thread
    for (; i + 3 * blockDim.x < block_vecs; i += 4 * blockDim.x) {
        const uint4 a = from[i], b = from[i + blockDim.x], c = from[i + 2 * blockDim.x],
                    d = from[i + 3 * blockDim.x];
        to[i] = a;
        to[i + blockDim.x] = b;
        to[i + 2 * blockDim.x] = c;
        to[i + 3 * blockDim.x] = d;
    }
    for (; i < block_vecs; i += blockDim.x) to[i] = from[i];
}

// grid (num_pairs, 2): copy whole blocks between two pools (blockIdx.y: K or
// V).  Either side may be pinned host memory; the same 16-byte vector loop as
// copy_blocks_kernel.  A dst named by another pair is skipped and flagged.
__global__ void __launch_bounds__(256)
    swap_blocks_kernel(const uint4 *__restrict__ src_k, const uint4 *__restrict__ src_v,
                       uint4 *__restrict__ dst_k, uint4 *__restrict__ dst_v, const int64_t *__restrict__ pairs,
                       int num_pairs, long long block_vecs, int src_num_blocks, int dst_num_blocks,
                       int32_t *status) {
    const int pidx = blockIdx.x;
    const int64_t src = pairs[2 * pidx], dst = pairs[2 * pidx + 1];
    __shared__ int conflict;
    if (threadIdx.x == 0) conflict = 0;
    __syncthreads();
    if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_status(status, PA_STATUS_BAD_PAIR);
        return;
    }
    for (int j = threadIdx.x; j < num_pairs; j += blockDim.x)
        if (j != pidx && pairs[2 * j + 1] == dst) conflict = 1;
    __syncthreads();
    if (conflict) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_status(status, PA_STATUS_BAD_PAIR);
        return;
    }
    const uint4 *from = (blockIdx.y == 0 ? src_k : src_v) + src * block_vecs;
    uint4 *to = (blockIdx.y == 0 ? dst_k : dst_v) + dst * block_vecs;
    long long i = threadIdx.x;
    for (; i + 3 * blockDim.x < block_vecs; i += 4 * blockDim.x) {
        const uint4 a = from[i], b = from[i + blockDim.x], c = from[i + 2 * blockDim.x],
                    d = from[i + 3 * blockDim.x];
        to[i] = a;
        to[i + blockDim.x] = b;
        to[i + 2 * blockDim.x] = c;
        to[i + 3 * blockDim.x] = d;
    }
    for (; i < block_vecs; i += blockDim.x) to[i] = from[i];
}

// One thread waits on a fresh barrier that no one arrives at; the bounded wait
// must give up and report it.
__global__ void wait_timeout_selftest_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(b, 0, limit_ns)) flag_status(status, PA_STATUS_WAIT_TIMEOUT);
}

}  // namespace pa

namespace {
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int elem_bytes(int dtype) { return dtype == PA_F32 ? 4 : (dtype == PA_BF16 ? 2 : 0); }

// True when the device can address `p`: device or managed memory, or pinned
// host memory with a device mapping equal to the host pointer (unified
// addressing).  Pageable host memory is refused rather than risked.
bool device_addressable(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}
}  // namespace

extern "C" int pa_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                                    const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                    int head_dim, int block_size, int num_blocks, int dtype,
                                    int32_t *dev_status, void *stream) {
    PaTraceRange trace("pa_reshape_and_cache");
    const int eb = elem_bytes(dtype);
    if (eb == 0) return pa_fail(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: bad dtype");
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: bad sizes");
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: null pointer");
    if ((head_dim * eb) % 16 != 0)
        return pa_fail(PA_ERR_UNSUPPORTED, "pa_reshape_and_cache: head_dim * element size must be a multiple of 16 bytes");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: misaligned pointer");
    const int row_vecs = head_dim * eb / 16;
    pa::reshape_and_cache_kernel<<<num_tokens, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), slot_mapping, num_kv_heads, row_vecs, block_size,
        static_cast<long long>(num_blocks) * block_size, dev_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, cudaGetErrorString(e));
    return PA_OK;
}

extern "C" int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs, int num_pairs,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype,
                              int32_t *dev_status, void *stream) {
    PaTraceRange trace("pa_copy_blocks");
    const int eb = elem_bytes(dtype);
    if (eb == 0) return pa_fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: bad dtype");
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: bad sizes");
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !src_dst_pairs) return pa_fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: null pointer");
    const long long block_bytes = static_cast<long long>(num_kv_heads) * block_size * head_dim * eb;
    if (block_bytes % 16 != 0)
        return pa_fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks: block bytes must be a multiple of 16");
    if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: misaligned pointer");
    dim3 grid(num_pairs, 2);
    pa::copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), src_dst_pairs, num_pairs,
        block_bytes / 16, num_blocks, dev_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, cudaGetErrorString(e));
    return PA_OK;
}

extern "C" int pa_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                              const int64_t *src_dst_pairs, int num_pairs, int src_num_blocks, int dst_num_blocks,
                              int num_kv_heads, int head_dim, int block_size, int dtype, int32_t *dev_status,
                              void *stream) {
    PaTraceRange trace("pa_swap_blocks");
    const int eb = elem_bytes(dtype);
    if (eb == 0) return pa_fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: bad dtype");
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || src_num_blocks <= 0 ||
        dst_num_blocks <= 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: bad sizes");
    if (num_pairs == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !src_dst_pairs)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: null pointer");
    if (src_k == dst_k || src_v == dst_v)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: source and destination pools must differ (use pa_copy_blocks)");
    const long long block_bytes = static_cast<long long>(num_kv_heads) * block_size * head_dim * eb;
    if (block_bytes % 16 != 0) return pa_fail(PA_ERR_UNSUPPORTED, "pa_swap_blocks: block bytes must be a multiple of 16");
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v) ||
        (reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: misaligned pointer");
    if (!device_addressable(src_k) || !device_addressable(src_v) || !device_addressable(dst_k) ||
        !device_addressable(dst_v) || !device_addressable(src_dst_pairs))
        return pa_fail(PA_ERR_INVALID_ARG,
                       "pa_swap_blocks: every pool and the pair list must be device memory or pinned host memory");
    dim3 grid(num_pairs, 2);
    pa::swap_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(src_k), static_cast<const uint4 *>(src_v), static_cast<uint4 *>(dst_k),
        static_cast<uint4 *>(dst_v), src_dst_pairs, num_pairs, block_bytes / 16, src_num_blocks, dst_num_blocks,
        dev_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, cudaGetErrorString(e));
    return PA_OK;
}

extern "C" int pa_selftest_wait_timeout(int32_t *dev_status, int limit_us, void *stream) {
    if (!dev_status || limit_us < 1 || limit_us > 1000000)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_selftest_wait_timeout: need a status word and 1 <= limit_us <= 1e6");
    pa::wait_timeout_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
        dev_status, static_cast<uint64_t>(limit_us) * 1000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, cudaGetErrorString(e));
    return PA_OK;
}
