// Device and host helpers shared by the decode kernels' translation units
// (the tensor-core pass and the split-K merge in pa_decode.cu, the fp32-FMA
// pass in pa_decode_simt.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ uint8_t *align_1024(uint8_t *p) {
    uint32_t a = smem_addr(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}

// Context length of sequence s, clamped into [0, ctx_cap].
__device__ __forceinline__ int seq_len(const DecodeParams &p, int s) {
    int n = p.context_lens[s];
    return n < 0 ? 0 : (n > p.ctx_cap ? p.ctx_cap : n);
}

__device__ __forceinline__ int parts_of(int n, int P) { return n <= P ? 1 : (n + P - 1) / P; }

// Position of the walk over (sequence, partition) pairs: `base` is the global
// index of sequence `seq`'s first partition.
struct SeqCursor {
    int seq;
    long long base;
};

// Move the cursor forward to the sequence that owns global partition gp
// (32 sequences per step, warp-parallel).  False when gp is past the end.
static __device__ bool seek(SeqCursor &c, long long gp, const DecodeParams &p, int lane) {
    while (c.seq < p.num_seqs) {
        const int s = c.seq + lane;
        const int np = s < p.num_seqs ? parts_of(seq_len(p, s), p.partition_size) : 0;
        int incl = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        const unsigned hit = __ballot_sync(kFull, s < p.num_seqs && gp < c.base + incl);
        if (hit) {
            const int L = __ffs(hit) - 1;
            c.base += __shfl_sync(kFull, incl - np, L);
            c.seq += L;
            return true;
        }
        c.base += __shfl_sync(kFull, incl, 31);
        c.seq += 32;
    }
    return false;
}

__device__ __forceinline__ void store4(float *dst, float4 v) { *reinterpret_cast<float4 *>(dst) = v; }

__device__ __forceinline__ void store4(__nv_bfloat16 *dst, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    memcpy(&u.x, &lo, 4);
    memcpy(&u.y, &hi, 4);
    *reinterpret_cast<uint2 *>(dst) = u;
}

// Merge the NW per-warp softmax states held in shared memory (each warp's
// region starts with float O[16][HD + kEpiPad], then M[16], then L[16]) and
// store either the final rows or the item's partial.
template <typename OutT, int HD, int NW = kWarps>
__device__ void merge_and_store(const uint8_t *smem, int warp_bytes, const DecodeParams &p, int seq,
                                int part, int qh0, int rows, bool single) {
    constexpr int LD = HD + kEpiPad;
    constexpr int Q4 = HD / 4;
    for (int task = threadIdx.x; task < rows * Q4; task += blockDim.x) {
        const int r = task / Q4, d = (task % Q4) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float *em = reinterpret_cast<const float *>(smem + w * warp_bytes) + 16 * LD;
            M = fmaxf(M, em[r]);
        }
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float *eo = reinterpret_cast<const float *>(smem + w * warp_bytes);
                const float f = exp2f(eo[16 * LD + r] - M);
                L += f * eo[16 * LD + 16 + r];
                const float4 v = *reinterpret_cast<const float4 *>(eo + r * LD + d);
                acc.x += f * v.x;
                acc.y += f * v.y;
                acc.z += f * v.z;
                acc.w += f * v.w;
            }
        }
        const int qh = qh0 + r;
        if (single) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
            OutT *o = static_cast<OutT *>(p.out) + ((long long)seq * p.num_q_heads + qh) * HD + d;
            store4(o, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
        } else {
            const long long idx = ((long long)seq * p.max_parts + part) * p.num_q_heads + qh;
            store4(p.part_acc + idx * HD + d, acc);
            if (d == 0) *reinterpret_cast<float2 *>(p.part_ml + idx * 2) = make_float2(M, L);
        }
    }
}

// Describes the item a CTA is working on.
struct Item {
    int seq, part, kvh, ht, qh0, rows, n;
    int tok_begin, tok_end, nchunks;
    bool single;
};

__device__ __forceinline__ bool next_item(Item &it, SeqCursor &cur, long long item,
                                          const DecodeParams &p, int tile_rows, int lane) {
    const int T = p.num_kv_heads * p.head_tiles;
    const long long gp = item / T;
    if (!seek(cur, gp, p, lane)) return false;
    const int r = static_cast<int>(item % T);
    const int ht = r % p.head_tiles;
    it.seq = cur.seq;
    it.part = static_cast<int>(gp - cur.base);
    it.kvh = r / p.head_tiles;
    it.ht = ht;
    it.qh0 = it.kvh * p.group + ht * tile_rows;
    it.rows = min(tile_rows, p.group - ht * tile_rows);
    const int raw = p.context_lens[it.seq];
    if (threadIdx.x == 0 && r == 0 && it.part == 0 && (raw < 0 || raw > p.ctx_cap))
        flag_status(p.status, PA_STATUS_BAD_CONTEXT_LEN);
    const int n = seq_len(p, it.seq);
    it.n = n;
    it.tok_begin = it.part * p.partition_size;
    it.tok_end = min(n, it.tok_begin + p.partition_size);
    const int ntok = max(0, it.tok_end - it.tok_begin);
    it.nchunks = (ntok + kChunk - 1) / kChunk;
    it.single = n <= p.partition_size;
    return true;
}

// Physical location of this warp's k-th chunk of the item, as a row of the
// [num_blocks * Hkv * block_size, head_dim] view of a cache; an invalid block
// id gives -1 and sets a flag (the passes then load rows past the view, which
// TMA fills with zeros).
template <int NW = kWarps>
__device__ __forceinline__ int chunk_row(const DecodeParams &p, const Item &it, int warp, int k) {
    const int c = warp + NW * k;
    const int tok = it.tok_begin + c * kChunk;
    const int phys = p.block_tables[(long long)it.seq * p.max_blocks_per_seq + tok / p.block_size];
    if (phys < 0 || phys >= p.num_blocks) {
        flag_status(p.status, PA_STATUS_BAD_BLOCK_ID);
        return -1;
    }
    return static_cast<int>(((long long)phys * p.num_kv_heads + it.kvh) * p.block_size +
                            tok % p.block_size);
}

// The new token of a fused cache write, as one item sees it: the item's chunk
// that holds position n - 1 (or -1), the row inside that chunk, and the row of
// the [num_blocks * Hkv * block_size, head_dim] cache view to write.  Only the
// last partition holds the new token; a slot that is not the slot of position
// n - 1 is flagged once (KV head 0, head tile 0) and ignored.
struct NewToken {
    int chunk, row;
    long long cache_row;
};

__device__ __forceinline__ NewToken new_token(const DecodeParams &p, const Item &it) {
    NewToken t{-1, 0, -1};
    if (!p.k_new || it.n <= 0 || it.tok_end != it.n) return t;
    const int64_t slot = p.slot_mapping[it.seq];
    if (slot < 0) return t;
    const int pos = it.n - 1;
    const int phys = p.block_tables[(long long)it.seq * p.max_blocks_per_seq + pos / p.block_size];
    if (phys < 0 || phys >= p.num_blocks || slot != (int64_t)phys * p.block_size + pos % p.block_size) {
        if (threadIdx.x == 0 && it.kvh == 0 && it.ht == 0) flag_status(p.status, PA_STATUS_BAD_SLOT);
        return t;
    }
    t.chunk = (pos - it.tok_begin) / kChunk;
    t.row = (pos - it.tok_begin) % kChunk;
    t.cache_row = ((long long)phys * p.num_kv_heads + it.kvh) * p.block_size + pos % p.block_size;
    return t;
}

// Work counter of the partition pass (one 64-bit word): hand-outs in the low
// half, finished CTAs in the high half.  Every CTA makes all its hand-out
// requests before it reports finishing, so when the last CTA reports, no
// request is left and the word can go back to zero for the next launch.
__device__ __forceinline__ long long next_handout(unsigned long long *ctr) {
    return static_cast<long long>(atomicAdd(ctr, 1ull) & 0xffffffffull);
}

__device__ __forceinline__ void finish_handouts(unsigned long long *ctr) {
    const unsigned long long before = atomicAdd(ctr, 1ull << 32);
    if ((before >> 32) == gridDim.x - 1u) atomicExch(ctr, 0ull);
}

// The per-partition pass on plain fp32 FMAs (fp32 inputs, or bf16 on request),
// defined in pa_decode_simt.cu.  Enqueues one launch on `st`.
int launch_simt_pass(const DecodeParams &p, const void *k_cache, const void *v_cache, bool f32, int head_dim,
                     long long items, int dev, cudaStream_t st);

// ------------------------------------------------------- host helpers ---
namespace host {

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

inline long long l2_bytes(int dev) {
    static std::atomic<long long> cache[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return 0;
    long long b = cache[dev].load(std::memory_order_relaxed);
    if (b == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
        b = v;
        cache[dev].store(b, std::memory_order_relaxed);
    }
    return b;
}

inline int sm_count(int dev) {
    static std::atomic<int> cache[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Per-kernel launch facts: dynamic smem set once, occupancy cached per device
// (guarded, so concurrent first calls from several host threads are safe).
struct KernelSlot {
    int smem = 0;
    int occupancy[kMaxDevices] = {0};
    std::mutex mu;
};

template <typename K>
int ensure_kernel(K kernel, KernelSlot &slot, int smem, int dev, int threads = kWarps * 32) {
    if (dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(slot.mu);
    if (slot.occupancy[dev] == 0) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return 0;
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess ||
            occ <= 0)
            return 0;
        slot.smem = smem;
        slot.occupancy[dev] = occ;
    }
    return slot.occupancy[dev];
}

// Tensor map of a cache seen as [rows][hd] (rows = num_blocks * Hkv *
// block_size), boxes of kChunk rows x 128 bytes (64 bf16 or 32 fp32 values)
// with the 128-byte swizzle; rows past the end read as zeros.
inline bool make_map(CUtensorMap *map, const void *base, long long rows, int hd, bool f32 = false) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const int elem = f32 ? 4 : 2;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(hd) * elem};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem), static_cast<cuuint32_t>(kChunk)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Launch a partition pass as a programmatic dependent of whatever kernel
// precedes it in the stream: its CTAs may be scheduled while that kernel's last
// CTAs finish, and wait in griddep_wait() before their first read of global
// memory.  After a copy or a kernel that triggers nothing it simply starts
// when that work is done.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), int grid, int threads, int smem, cudaStream_t st,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace host
}  // namespace pa
