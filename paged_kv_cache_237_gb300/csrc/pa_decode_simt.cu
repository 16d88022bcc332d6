// Paged decode attention, per-partition pass on plain fp32 FMAs (sm_103a).
//
// What is computed is the same as in pa_decode.cu ("PagedAttention",
// robocikowo.com, "Jak dziala" and "Komponenty": the kernel reads each
// sequence's cache through its block table; "PagedAttention et RadixAttention
// : parlons de KV Cache", aitalk.it, "PagedAttention : la memoire comme un
// systeme d'exploitation", step two).  This pass serves fp32 caches, and bf16
// caches when the caller asks for fp32 products throughout.  Like the
// tensor-core pass it is bound by HBM bandwidth, so its arithmetic is laid out
// to stay off the critical path:
//
//  - Staging.  Each warp owns a ring of stages; a stage is one 16-token chunk
//    of K and V, loaded by 2-D TMA in boxes of 16 rows x 128 bytes with the
//    128-byte swizzle (16-byte granule g of row r lands at granule g ^ (r & 7)
//    of that row's 128-byte line).  Loads carry an L2 evict-first hint: each
//    K/V row is read once per step.
//  - q.K: lane = (token, half of head_dim).  Each lane dots its token's half
//    row against q, read from shared memory as a broadcast, for every query
//    head of the tile, and one shuffle adds the two halves.  No per-token warp
//    reduction: the swizzle puts the 8 tokens a quarter-warp reads on 8
//    different bank groups.  Products use Blackwell's packed fp32x2 FMA
//    (each half of the pair rounded as fmaf would), accumulating even and odd
//    elements separately.
//  - Online softmax per chunk: one max over the 16 token lanes per head, the
//    probabilities written to shared memory.
//  - p.V: lane = (16-byte granule of head_dim, token slice).  Each lane reads
//    its granule of every token row (a permutation of one 128-byte line per
//    quarter-warp, so no bank conflict) and the tile's probabilities of that
//    token as a broadcast (stored twice, as a packed multiplier), and
//    accumulates in fp32 with packed FMAs.
//  - Work items, the end-of-item merge of the warps' states and the split-K
//    layout are those of the tensor-core pass (pa_decode_common.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "pa_decode_common.cuh"

// Launch shapes, written as warps per CTA x 100 + ring depth per warp x 10 +
// CTAs per SM.  A stage is 16 tokens of K and V: 16 KB for fp32 at head_dim
// 128.  The pass is bound by issue latency before bandwidth, so it wants many
// warps and several independent CTAs per SM (one CTA's item start and merge
// then overlap the others' streams): fp32 at head_dim 128 runs 3 CTAs of 4
// warps with one stage each (measured on the GQA-8 batch: 0.94 of the copy
// peak, against 0.68 with 1 CTA of 4 warps x 3 stages and 0.85 with 3 CTAs of
// 2 warps x 2 stages).
#ifndef PA_SIMT_SHAPE_F32_128
#define PA_SIMT_SHAPE_F32_128 413
#endif
#ifndef PA_SIMT_SHAPE_F32_64
#define PA_SIMT_SHAPE_F32_64 414
#endif
#ifndef PA_SIMT_SHAPE_BF16_128
#define PA_SIMT_SHAPE_BF16_128 423
#endif
#ifndef PA_SIMT_SHAPE_BF16_64
#define PA_SIMT_SHAPE_BF16_64 434
#endif

namespace pa {
namespace {

template <int CODE>
struct Shape {
    static constexpr int NW = CODE / 100, NSTAGE = CODE / 10 % 10, CPS = CODE % 10;
};
template <typename T, int HD>
struct SimtShape;
template <>
struct SimtShape<float, 128> : Shape<PA_SIMT_SHAPE_F32_128> {};
template <>
struct SimtShape<float, 64> : Shape<PA_SIMT_SHAPE_F32_64> {};
template <>
struct SimtShape<__nv_bfloat16, 128> : Shape<PA_SIMT_SHAPE_BF16_128> {};
template <>
struct SimtShape<__nv_bfloat16, 64> : Shape<PA_SIMT_SHAPE_BF16_64> {};

constexpr int kSimtTile = 8;   // query heads per work item (at most)

// One 16-byte granule of a staged row, widened to fp32 as pairs of adjacent
// elements (the operands of the packed fp32x2 FMAs below).
__device__ __forceinline__ void unpack(const uint4 &raw, float2 (&f)[2]) {
    f[0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
    f[1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
}

__device__ __forceinline__ void unpack(const uint4 &raw, float2 (&f)[4]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)   // a bf16 value is the upper half of the fp32 with the same bits
        f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T, int HD, int HT, int NW, int NSTAGE>
struct SimtLayout {
    static constexpr int E = static_cast<int>(sizeof(T));
    static constexpr int VEC = 16 / E;                 // elements per 16-byte granule
    static constexpr int GPR = HD / VEC;               // granules per row
    static constexpr int NBOX = HD * E / 128;          // 128-byte TMA boxes per row
    static constexpr int BOX_W = 128 / E;              // elements per box row
    static constexpr int BOX_BYTES = kChunk * 128;
    static constexpr int PAGE_BYTES = NBOX * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * PAGE_BYTES; // K, then V
    static constexpr int WARP_BYTES = NSTAGE * STAGE_BYTES;
    static constexpr int BAR_BYTES = (NW * NSTAGE * 8 + 15) / 16 * 16;
    static constexpr int QLD = HD + 8;                 // q row stride (floats)
    static constexpr int QHALF = HD / 2 + 4;           // where a q row's second half starts
    static constexpr int Q_BYTES = HT * QLD * 4;
    static constexpr int P_BYTES = NW * kChunk * HT * 8;   // each probability twice (a packed pair)
    static constexpr int SMEM = NW * WARP_BYTES + BAR_BYTES + Q_BYTES + P_BYTES + 1024;
    // Chunks of one item per warp, at most (partitions of up to 4096 tokens),
    // and the 32-wide register slots that hold their rows.
    static constexpr int MAX_CHUNKS = (4096 / kChunk + NW - 1) / NW;
    static constexpr int RSLOTS = (MAX_CHUNKS + 31) / 32;
};

template <typename T, int HD, int HT, int NW, int NSTAGE, int CPS>
__global__ void __launch_bounds__(NW * 32, CPS)
    decode_simt_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const DecodeParams p) {
    using Lay = SimtLayout<T, HD, HT, NW, NSTAGE>;
    constexpr int VEC = Lay::VEC, GPR = Lay::GPR, NBOX = Lay::NBOX;
    constexpr int BOX_BYTES = Lay::BOX_BYTES, PAGE_BYTES = Lay::PAGE_BYTES, STAGE_BYTES = Lay::STAGE_BYTES;
    constexpr int WARP_BYTES = Lay::WARP_BYTES, QLD = Lay::QLD, QHALF = Lay::QHALF;
    constexpr int KG = GPR / 2;     // granules per lane in q.K
    constexpr int TS = 32 / GPR;    // token slices in p.V
    constexpr int LD = HD + kEpiPad;
    static_assert(GPR <= 32 && 32 % GPR == 0, "a warp covers a row in whole granules");
    static_assert(WARP_BYTES >= (16 * LD + 32) * 4, "epilogue tile must fit in a warp's stages");
    static_assert(HT == 1 || HT == 2 || HT == 4 || HT == 8, "head tile");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *wbuf = smem + warp * WARP_BYTES;
    const uint32_t wbuf_s = smem_addr(wbuf);
    const uint32_t bar_s = smem_addr(smem + NW * WARP_BYTES) + warp * NSTAGE * 8;
    float *q_s = reinterpret_cast<float *>(smem + NW * WARP_BYTES + Lay::BAR_BYTES);
    float *p_s = q_s + HT * QLD + warp * kChunk * HT * 2;

    if (lane == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(bar_s + 8 * s, 1);
        fence_mbar_init();
        if (warp == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
    }
    __syncwarp();

    uint32_t n_issued = 0, n_done = 0;
    bool failed = false;
    SeqCursor cur{0, 0};
    const int oob_row = p.total_rows;
    const uint64_t kv_policy = l2_evict_first_policy();
    const int tok = lane & 15, half = lane >> 4;      // q.K roles
    const int dg = lane % GPR, ts = lane / GPR;       // p.V roles
    // Launched as a programmatic dependent: from here on the CTA reads what
    // earlier work in the stream wrote (q, tables, caches, the work counter).
    griddep_wait();

    // Work items as in the tensor-core pass: the first is blockIdx.x, later
    // ones come from the work counter (one fetched ahead) when there is one,
    // else every gridDim.x-th.
    __shared__ long long s_next[2];
    const bool dynamic = p.work_ctr != nullptr;
    long long ahead = 0;
    if (dynamic && threadIdx.x == 0) ahead = gridDim.x + next_handout(p.work_ctr);
    int nb = 0;
    for (long long item = blockIdx.x;;) {
        Item it;
        if (!next_item(it, cur, item, p, kSimtTile, lane)) break;
        const int my_n = it.nchunks > warp ? (it.nchunks - warp + NW - 1) / NW : 0;

        // Rows of this warp's chunks: slot j of lane i holds chunk i + 32 j.
        int rows[Lay::RSLOTS];
#pragma unroll
        for (int j = 0; j < Lay::RSLOTS; ++j) {
            rows[j] = oob_row;
            if (lane + 32 * j < my_n) {
                const int r = chunk_row<NW>(p, it, warp, lane + 32 * j);
                rows[j] = r < 0 ? oob_row : r;
            }
        }

        auto issue = [&](int k) {
            int rv = rows[0];
#pragma unroll
            for (int j = 1; j < Lay::RSLOTS; ++j)
                if ((k >> 5) == j) rv = rows[j];
            const int row = __shfl_sync(kFull, rv, k & 31);
            if (failed) return;
            if (lane == 0) {
                const int s = n_issued % NSTAGE;
                const uint32_t dst = wbuf_s + s * STAGE_BYTES, bar = bar_s + 8 * s;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, STAGE_BYTES);
#pragma unroll
                for (int b = 0; b < NBOX; ++b) {
                    tma_load_2d_hint(dst + b * BOX_BYTES, &tmK, b * Lay::BOX_W, row, bar, kv_policy);
                    tma_load_2d_hint(dst + PAGE_BYTES + b * BOX_BYTES, &tmV, b * Lay::BOX_W, row, bar, kv_policy);
                }
            }
            ++n_issued;
        };

        const int pro = my_n < NSTAGE ? my_n : NSTAGE;
        for (int k = 0; k < pro; ++k) issue(k);

        // q of the tile, widened and pre-scaled by scale * log2(e), rows past
        // the tile's heads zero.  The previous item's last barrier means no
        // warp still reads the old values.
        {
            const T *qb = static_cast<const T *>(p.q) + ((long long)it.seq * p.num_q_heads + it.qh0) * HD;
            for (int i = threadIdx.x; i < HT * HD; i += NW * 32) {
                const int h = i / HD, d = i % HD;
                const float v = h < it.rows ? to_f32(qb[h * HD + d]) * p.scale_log2 : 0.f;
                q_s[h * QLD + d + (d >= HD / 2 ? 4 : 0)] = v;
            }
        }
        const NewToken ntok = new_token(p, it);
        __syncthreads();

        float2 acc[HT][VEC / 2];   // this lane's granule of each head's output, as pairs
        float m[HT], l[HT];
#pragma unroll
        for (int h = 0; h < HT; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int v = 0; v < VEC / 2; ++v) acc[h][v] = make_float2(0.f, 0.f);
        }

        for (int k = 0; k < my_n; ++k) {
            const int s = n_done % NSTAGE;
            const uint32_t parity = (n_done / NSTAGE) & 1u;
            bool ok = !failed && mbar_wait_bounded(bar_s + 8 * s, parity);
            if (__any_sync(kFull, !ok)) {
                if (!failed && lane == 0) flag_status(p.status, PA_STATUS_WAIT_TIMEOUT);
                failed = true;
                break;
            }
            ++n_done;
            uint8_t *stage = wbuf + s * STAGE_BYTES;
            const uint8_t *Ks = stage;
            const uint8_t *Vs = stage + PAGE_BYTES;
            const int c = warp + NW * k;
            const int valid = min(kChunk, it.tok_end - (it.tok_begin + c * kChunk));
            if (c == ntok.chunk) {
                // Fused cache write: the new token's row goes into the staged
                // tile (whatever the copy read) and, once per (sequence, KV
                // head), into the caches.
                const long long src = ((long long)it.seq * p.num_kv_heads + it.kvh) * GPR;
                const uint4 *kn = static_cast<const uint4 *>(p.k_new) + src;
                const uint4 *vn = static_cast<const uint4 *>(p.v_new) + src;
                const int r = ntok.row;
                for (int i = lane; i < 2 * GPR; i += 32) {
                    const bool isv = i >= GPR;
                    const int g = isv ? i - GPR : i;
                    const uint4 val = isv ? vn[g] : kn[g];
                    *reinterpret_cast<uint4 *>(stage + (isv ? PAGE_BYTES : 0) + (g >> 3) * BOX_BYTES + r * 128 +
                                               (((g & 7) ^ (r & 7)) << 4)) = val;
                    if (it.ht == 0)
                        static_cast<uint4 *>(isv ? p.v_cache_w : p.k_cache_w)[ntok.cache_row * GPR + g] = val;
                }
                fence_proxy_async_smem();
                __syncwarp();
            }

            // s = q.K for this lane's token and half row, every head of the tile,
            // accumulated as (even, odd) element pairs by packed FMAs.
            float2 sc2[HT];
#pragma unroll
            for (int h = 0; h < HT; ++h) sc2[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < KG; ++j) {
                const int g = half * KG + j;
                const uint4 raw = *reinterpret_cast<const uint4 *>(Ks + (g >> 3) * BOX_BYTES + tok * 128 +
                                                                   (((g & 7) ^ (tok & 7)) << 4));
                float2 kv[VEC / 2];
                unpack(raw, kv);
                const float *qp = q_s + half * QHALF + j * VEC;
#pragma unroll
                for (int h = 0; h < HT; ++h) {
#pragma unroll
                    for (int v4 = 0; v4 < VEC; v4 += 4) {
                        const float4 qv = *reinterpret_cast<const float4 *>(qp + h * QLD + v4);
                        sc2[h] = __ffma2_rn(make_float2(qv.x, qv.y), kv[v4 / 2], sc2[h]);
                        sc2[h] = __ffma2_rn(make_float2(qv.z, qv.w), kv[v4 / 2 + 1], sc2[h]);
                    }
                }
            }

            // Online softmax, base 2 (q carries scale * log2 e).  Both halves
            // of the warp hold the same 16 scores, so m stays warp-uniform.
            float pr[HT], alpha[HT];
#pragma unroll
            for (int h = 0; h < HT; ++h) {
                const float part = sc2[h].x + sc2[h].y;
                float x = part + __shfl_xor_sync(kFull, part, 16);
                x = tok < valid ? x : -INFINITY;   // slots past the context may hold anything
                float mx = fmaxf(x, __shfl_xor_sync(kFull, x, 1));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                const float mn = fmaxf(m[h], mx);
                const float ref = mn == -INFINITY ? 0.f : mn;
                alpha[h] = exp2f(m[h] - ref);
                m[h] = mn;
                pr[h] = exp2f(x - ref);
                l[h] = l[h] * alpha[h] + pr[h];
            }
            {
                // p_s[token][head] holds each probability twice, the packed
                // multiplier of p.V; the two halves of the warp write half of
                // the heads each.
                float2 *pw = reinterpret_cast<float2 *>(p_s) + tok * HT;
                if constexpr (HT == 1) {
                    if (half == 0) pw[0] = make_float2(pr[0], pr[0]);
                } else {
#pragma unroll
                    for (int i = 0; i < HT / 2; ++i) {
                        const float v = half ? pr[HT / 2 + i] : pr[i];
                        pw[half * (HT / 2) + i] = make_float2(v, v);
                    }
                }
            }
            bool rescale = false;
#pragma unroll
            for (int h = 0; h < HT; ++h) rescale |= alpha[h] != 1.f;
            if (rescale) {
#pragma unroll
                for (int h = 0; h < HT; ++h)
#pragma unroll
                    for (int v = 0; v < VEC / 2; ++v)
                        acc[h][v] = __fmul2_rn(acc[h][v], make_float2(alpha[h], alpha[h]));
            }
            __syncwarp();

            // acc += p V: this lane's granule of every valid token of its slice.
            auto pv_token = [&](int t) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(Vs + (dg >> 3) * BOX_BYTES + t * 128 +
                                                                   (((dg & 7) ^ (t & 7)) << 4));
                float2 vv[VEC / 2];
                unpack(raw, vv);
                float2 pt[HT];
                const float2 *pp = reinterpret_cast<const float2 *>(p_s) + t * HT;
                if constexpr (HT >= 2) {
#pragma unroll
                    for (int h = 0; h < HT; h += 2) {
                        const float4 q4 = *reinterpret_cast<const float4 *>(pp + h);
                        pt[h] = make_float2(q4.x, q4.y);
                        pt[h + 1] = make_float2(q4.z, q4.w);
                    }
                } else {
                    pt[0] = pp[0];
                }
#pragma unroll
                for (int h = 0; h < HT; ++h)
#pragma unroll
                    for (int v = 0; v < VEC / 2; ++v) acc[h][v] = __ffma2_rn(pt[h], vv[v], acc[h][v]);
            };
            if (valid == kChunk) {
#pragma unroll
                for (int i = 0; i < kChunk / TS; ++i) pv_token(ts + i * TS);
            } else {
                for (int t = ts; t < valid; t += TS) pv_token(t);
            }
            __syncwarp();   // p_s and this stage are free again
            if (k + NSTAGE < my_n) issue(k + NSTAGE);
        }

        // Epilogue: sum l over the 16 token lanes and acc over the token
        // slices, then publish this warp's state in its (now idle) stages.
#pragma unroll
        for (int h = 0; h < HT; ++h) {
            l[h] += __shfl_xor_sync(kFull, l[h], 1);
            l[h] += __shfl_xor_sync(kFull, l[h], 2);
            l[h] += __shfl_xor_sync(kFull, l[h], 4);
            l[h] += __shfl_xor_sync(kFull, l[h], 8);
        }
#pragma unroll
        for (int o = GPR; o < 32; o <<= 1)
#pragma unroll
            for (int h = 0; h < HT; ++h)
#pragma unroll
                for (int v = 0; v < VEC / 2; ++v) {
                    acc[h][v].x += __shfl_xor_sync(kFull, acc[h][v].x, o);
                    acc[h][v].y += __shfl_xor_sync(kFull, acc[h][v].y, o);
                }
        {
            float *eo = reinterpret_cast<float *>(wbuf);
            if (ts == 0) {
#pragma unroll
                for (int h = 0; h < HT; ++h)
#pragma unroll
                    for (int v = 0; v < VEC / 2; v += 2)
                        *reinterpret_cast<float4 *>(eo + h * LD + dg * VEC + 2 * v) =
                            make_float4(acc[h][v].x, acc[h][v].y, acc[h][v + 1].x, acc[h][v + 1].y);
            }
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    eo[16 * LD + h] = h < HT ? m[h < HT ? h : 0] : -INFINITY;
                    eo[16 * LD + 16 + h] = h < HT ? l[h < HT ? h : 0] : 0.f;
                }
            }
        }
        if (threadIdx.x == 0) s_next[nb] = dynamic ? ahead : item + gridDim.x;
        __syncthreads();
        merge_and_store<T, HD, NW>(smem, WARP_BYTES, p, it.seq, it.part, it.qh0, it.rows, it.single);
        fence_proxy_async_smem();
        __syncthreads();
        item = s_next[nb];
        nb ^= 1;
        if (dynamic && threadIdx.x == 0) ahead = gridDim.x + next_handout(p.work_ctr);
    }
    // No more items for this CTA: the merge launch may start taking its place.
    griddep_launch_dependents();
    if (dynamic && threadIdx.x == 0) finish_handouts(p.work_ctr);

    // A wait gave up: let copies still in flight land before the CTA exits.
    if (failed && lane == 0) {
        for (uint32_t gi = n_done; gi < n_issued; ++gi)
            mbar_wait_bounded(bar_s + 8 * (gi % NSTAGE), (gi / NSTAGE) & 1u);
    }
}

template <typename T, int HD, int HT>
int launch_one(const DecodeParams &p, const void *k_cache, const void *v_cache, long long items, int dev,
               cudaStream_t st) {
    using S = SimtShape<T, HD>;
    using Lay = SimtLayout<T, HD, HT, S::NW, S::NSTAGE>;
    static host::KernelSlot slot;
    auto kernel = decode_simt_kernel<T, HD, HT, S::NW, S::NSTAGE, S::CPS>;
    const int occ = host::ensure_kernel(kernel, slot, Lay::SMEM, dev, S::NW * 32);
    if (occ == 0) return pa_fail(PA_ERR_CUDA, "pa_decode: cannot configure the fp32-FMA kernel");
    CUtensorMap mk, mv;
    const bool f32 = sizeof(T) == 4;
    if (!host::make_map(&mk, k_cache, p.total_rows, HD, f32) || !host::make_map(&mv, v_cache, p.total_rows, HD, f32))
        return pa_fail(PA_ERR_CUDA, "pa_decode: cuTensorMapEncodeTiled failed");
    const long long cap = static_cast<long long>(host::sm_count(dev)) * occ;
    const int grid = static_cast<int>(items < cap ? items : cap);
    const cudaError_t e = host::launch_dependent(kernel, grid, S::NW * 32, Lay::SMEM, st, mk, mv, p);
    if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, cudaGetErrorString(e));
    return PA_OK;
}

template <typename T, int HD>
int launch_tile(const DecodeParams &p, const void *k_cache, const void *v_cache, long long items, int dev,
                cudaStream_t st) {
    if (p.tile_rows <= 1) return launch_one<T, HD, 1>(p, k_cache, v_cache, items, dev, st);
    if (p.tile_rows <= 2) return launch_one<T, HD, 2>(p, k_cache, v_cache, items, dev, st);
    if (p.tile_rows <= 4) return launch_one<T, HD, 4>(p, k_cache, v_cache, items, dev, st);
    return launch_one<T, HD, 8>(p, k_cache, v_cache, items, dev, st);
}

}  // namespace

int launch_simt_pass(const DecodeParams &p, const void *k_cache, const void *v_cache, bool f32, int head_dim,
                     long long items, int dev, cudaStream_t st) {
    if (p.tile_rows < 1 || p.tile_rows > kSimtTile)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: head tile out of range for the fp32-FMA kernel");
    if (f32)
        return head_dim == 128 ? launch_tile<float, 128>(p, k_cache, v_cache, items, dev, st)
                               : launch_tile<float, 64>(p, k_cache, v_cache, items, dev, st);
    return head_dim == 128 ? launch_tile<__nv_bfloat16, 128>(p, k_cache, v_cache, items, dev, st)
                           : launch_tile<__nv_bfloat16, 64>(p, k_cache, v_cache, items, dev, st);
}

}  // namespace pa
