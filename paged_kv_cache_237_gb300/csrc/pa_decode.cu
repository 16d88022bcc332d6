// Paged decode attention for sm_103a.
//
// What is computed: for each sequence and query head, attention of the one
// decode query over the sequence's cached K/V, which live in fixed-size
// physical blocks reached through the sequence's block table ("PagedAttention",
// robocikowo.com, "Jak dziala" and "Komponenty": a custom kernel reads the
// non-contiguous cache through the block table; "PagedAttention et
// RadixAttention : parlons de KV Cache", aitalk.it, "PagedAttention : la
// memoire comme un systeme d'exploitation", step two).  The path is bound by
// HBM bandwidth ("PagedAttention", robocikowo.com, "Zlozonosc obliczeniowa").
//
// Work decomposition.  A work item is (sequence, context partition, KV head,
// query-head tile).  A persistent grid walks the items in order, each CTA
// taking the next unclaimed item from a device counter (bf16 path with a
// workspace); a CTA owns an item and its 4 warps split the item's 16-token
// chunks round-robin.  Each warp runs its own ring of NSTAGE shared-memory
// stages, filled by TMA and tracked by one mbarrier per stage, so the main
// loop needs no CTA-wide barrier.  At the end of the item the warps' partial
// softmax states (max, sum, unnormalised output) are merged through shared
// memory; single-partition sequences write the final output, the others write
// a partial that the reduce kernel merges.
//
// bf16 path: each 16-token chunk of K and V arrives as 2-D TMA boxes of
// 16 rows x 64 elements with the 128-byte swizzle, which makes the ldmatrix
// reads below bank-conflict free.  The boxes are loaded under an L2
// evict-first policy: each K/V row is read once per step, and the split-K
// partials written meanwhile then stay in L2.  The query-head group (up to 16
// heads) is the M dimension of mma.m16n8k16: S = Q K^T (tokens are N), the fp32
// probabilities, split into a bf16 high part and a bf16 residual, feed
// O += P_hi V + P_lo V directly from registers (two MMAs keep ~16 bits of p).
// fp32 inputs (and bf16 on request) take a pass on plain fp32 FMAs instead,
// pa_decode_simt.cu; the split-K merge below serves both.
// Fused cache write (optional): the warp whose chunk holds a sequence's new
// last token copies that row into its staged tile, and the CTA of query-head
// tile 0 writes it to the caches, so one launch both writes and attends.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pa_decode_common.cuh"

namespace pa {

// ------------------------------------------------------------ bf16 path ---
// Launch shape per head_dim: ring depth per warp and the CTAs per SM the
// kernel is built for (its launch bounds hold registers to what that needs).
// hd128: 2 stages of 8 KB (64 KB of stages per CTA), 3 CTAs per SM (shared
// memory, and 168 registers x 128 threads x 3); with the dynamic item hand-out
// this beats 3 stages at 2 CTAs per SM on every batch measured.  hd64: 3
// stages of 4 KB (48 KB per CTA), 4 CTAs per SM, 3-6 % faster than 4 stages at
// 3 CTAs per SM.
template <int HD>
constexpr int bf16_stages() { return HD == 128 ? 2 : 3; }
template <int HD>
constexpr int bf16_ctas_per_sm() { return HD == 128 ? 3 : 4; }

template <int HD, int NSTAGE, bool ROWS16>
__global__ void __launch_bounds__(kWarps * 32, bf16_ctas_per_sm<HD>())
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
    constexpr int HALVES = HD / 64;              // 128-byte column slices per row
    constexpr int HALF_BYTES = kChunk * 128;     // one TMA box: 16 rows x 64 bf16
    constexpr int PAGE_BYTES = HALVES * HALF_BYTES;
    constexpr int STAGE_BYTES = 2 * PAGE_BYTES;  // K, then V
    constexpr int WARP_BYTES = NSTAGE * STAGE_BYTES;
    constexpr int KT = HD / 16;
    constexpr int NT = HD / 8;
    constexpr int LD = HD + kEpiPad;
    static_assert(WARP_BYTES >= (16 * LD + 32) * 4, "epilogue tile must fit in a warp's stages");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    uint8_t *wbuf = smem + warp * WARP_BYTES;
    const uint32_t wbuf_s = smem_addr(wbuf);
    const uint32_t bar_s = smem_addr(smem + kWarps * WARP_BYTES) + warp * NSTAGE * 8;

    if (lane == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(bar_s + 8 * s, 1);
        fence_mbar_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncwarp();

    uint32_t n_issued = 0, n_done = 0;
    bool failed = false;
    SeqCursor cur{0, 0};
    const int oob_row = p.total_rows;
    const uint64_t kv_policy = l2_evict_first_policy();
    // Launched as a programmatic dependent: everything above touched only this
    // CTA's registers and shared memory; from here on it reads what earlier
    // work in the stream wrote (q, tables, caches, the work counter).
    griddep_wait();

    // Work items: a CTA's first is blockIdx.x; later ones come from the work
    // counter in the workspace when there is one (a CTA that finishes early
    // takes more), else every gridDim.x-th.  Either way a CTA's items increase,
    // as the forward-only sequence cursor needs.  Thread 0 fetches the next
    // index one item ahead, so the atomic's latency hides behind the item.
    // s_next is double-buffered: the main loop has no CTA-wide barrier between
    // a warp's read of one entry and thread 0's next write to it.  The
    // counter's low 32 bits count hand-outs, its high 32 bits CTAs that have
    // finished; the last CTA to finish sets it back to zero.
    __shared__ long long s_next[2];
    const bool dynamic = p.work_ctr != nullptr;
    long long ahead = 0;
    if (dynamic && threadIdx.x == 0) ahead = gridDim.x + next_handout(p.work_ctr);
    int nb = 0;
    for (long long item = blockIdx.x;;) {
        Item it;
        if (!next_item(it, cur, item, p, 16, lane)) break;
        const int my_n = it.nchunks > warp ? (it.nchunks - warp + kWarps - 1) / kWarps : 0;

        // Rows of this warp's chunks: lane j holds chunks j and j + 32.
        int rowA = oob_row, rowB = oob_row;
        if (lane < my_n) {
            int r = chunk_row(p, it, warp, lane);
            rowA = r < 0 ? oob_row : r;
        }
        if (lane + 32 < my_n) {
            int r = chunk_row(p, it, warp, lane + 32);
            rowB = r < 0 ? oob_row : r;
        }

        auto issue = [&](int k) {
            const int row = __shfl_sync(kFull, k < 32 ? rowA : rowB, k & 31);
            if (failed) return;
            if (lane == 0) {
                const int s = n_issued % NSTAGE;
                const uint32_t dst = wbuf_s + s * STAGE_BYTES, bar = bar_s + 8 * s;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, STAGE_BYTES);
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    tma_load_2d_hint(dst + h * HALF_BYTES, &tmK, h * 64, row, bar, kv_policy);
                    tma_load_2d_hint(dst + PAGE_BYTES + h * HALF_BYTES, &tmV, h * 64, row, bar, kv_policy);
                }
            }
            ++n_issued;
        };

        // Q fragments (A operand), rows >= it.rows are zero.
        uint32_t qa[KT][4];
        {
            const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q) +
                                      ((long long)it.seq * p.num_q_heads + it.qh0) * HD;
            const bool lo_ok = g < it.rows, hi_ok = ROWS16 && (g + 8 < it.rows);
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                const int c0 = 16 * kk + 2 * t;
                qa[kk][0] = lo_ok ? *reinterpret_cast<const uint32_t *>(qb + g * HD + c0) : 0u;
                qa[kk][1] = hi_ok ? *reinterpret_cast<const uint32_t *>(qb + (g + 8) * HD + c0) : 0u;
                qa[kk][2] = lo_ok ? *reinterpret_cast<const uint32_t *>(qb + g * HD + c0 + 8) : 0u;
                qa[kk][3] = hi_ok ? *reinterpret_cast<const uint32_t *>(qb + (g + 8) * HD + c0 + 8) : 0u;
            }
        }

        const int pro = my_n < NSTAGE ? my_n : NSTAGE;
        for (int k = 0; k < pro; ++k) issue(k);
        const NewToken ntok = new_token(p, it);   // its loads overlap the copies in flight

        float o[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

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
            const uint32_t Ks = wbuf_s + s * STAGE_BYTES, Vs = Ks + PAGE_BYTES;
            const int tok0 = it.tok_begin + (warp + kWarps * k) * kChunk;
            const int valid = min(kChunk, it.tok_end - tok0);
            if (warp + kWarps * k == ntok.chunk) {
                // Fused cache write: put the new token's K/V row into the staged
                // tile (whatever the copy read) and, once per (sequence, KV
                // head), into the caches.
                constexpr int V16 = HD / 8;   // 16-byte pieces per row
                const long long src = ((long long)it.seq * p.num_kv_heads + it.kvh) * V16;
                const uint4 *kn = static_cast<const uint4 *>(p.k_new) + src;
                const uint4 *vn = static_cast<const uint4 *>(p.v_new) + src;
                uint8_t *st = wbuf + s * STAGE_BYTES;
                const int r = ntok.row;
                for (int i = lane; i < 2 * V16; i += 32) {
                    const bool isv = i >= V16;
                    const int c = isv ? i - V16 : i;
                    const uint4 val = isv ? vn[c] : kn[c];
                    *reinterpret_cast<uint4 *>(st + (isv ? PAGE_BYTES : 0) + (c >> 3) * HALF_BYTES + r * 128 +
                                               (((c & 7) ^ (r & 7)) << 4)) = val;
                    if (it.ht == 0)
                        static_cast<uint4 *>(isv ? p.v_cache_w : p.k_cache_w)[ntok.cache_row * V16 + c] = val;
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (valid < kChunk) {
                // Tokens past the context: zero their V rows so that p = 0
                // multiplies exact zeros (the slots may hold anything, NaN too).
                uint8_t *vg = wbuf + s * STAGE_BYTES + PAGE_BYTES;
                const int per_half = (kChunk - valid) * 8;
                for (int i = lane; i < HALVES * per_half; i += 32) {
                    const int h = i / per_half, rem = i % per_half;
                    *reinterpret_cast<uint4 *>(vg + h * HALF_BYTES + (valid + rem / 8) * 128 +
                                               (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }

            // S = Q K^T over the 16 tokens (two n-tiles of 8 tokens).
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                const int mi = lane >> 3;
                const int r = (lane & 7) + ((mi >> 1) << 3);
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    const int ch = 2 * kk + (mi & 1);
                    const uint32_t addr =
                        Ks + (ch >> 3) * HALF_BYTES + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(addr, b0, b1, b2, b3);
                    mma_bf16_16816(sc[0], qa[kk], b0, b1);
                    mma_bf16_16816(sc[1], qa[kk], b2, b3);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tok = 8 * nt + 2 * t + (j & 1);
                    sc[nt][j] = tok < valid ? sc[nt][j] * p.scale_log2 : -INFINITY;
                }

            // Online softmax, base 2.  Row g uses sc[.][0..1], row g + 8 sc[.][2..3].
            float mx_lo = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(kFull, mx_lo, 1));
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(kFull, mx_lo, 2));
            const float mn_lo = fmaxf(m_lo, mx_lo);
            const float ref_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
            const float alpha_lo = exp2f(m_lo - ref_lo);
            m_lo = mn_lo;
            float alpha_hi = 1.f, ref_hi = 0.f;
            if (ROWS16) {
                float mx_hi = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(kFull, mx_hi, 1));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(kFull, mx_hi, 2));
                const float mn_hi = fmaxf(m_hi, mx_hi);
                ref_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
                alpha_hi = exp2f(m_hi - ref_hi);
                m_hi = mn_hi;
            }
            // Probabilities in fp32, then split as p = hi + lo with both parts
            // bf16, so that P V on bf16 MMAs keeps ~16 significant bits of p.
            float pr[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                pr[nt][0] = exp2f(sc[nt][0] - ref_lo);
                pr[nt][1] = exp2f(sc[nt][1] - ref_lo);
                pr[nt][2] = ROWS16 ? exp2f(sc[nt][2] - ref_hi) : 0.f;
                pr[nt][3] = ROWS16 ? exp2f(sc[nt][3] - ref_hi) : 0.f;
            }
            l_lo = l_lo * alpha_lo + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
            if (ROWS16) l_hi = l_hi * alpha_hi + ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
            uint32_t pa[4], pb[4];
            {
                // A-fragment order: (row g, tok 2t..), (row g+8, tok 2t..),
                // (row g, tok 8+2t..), (row g+8, tok 8+2t..)
                const float *src[4][2] = {{&pr[0][0], &pr[0][1]}, {&pr[0][2], &pr[0][3]},
                                          {&pr[1][0], &pr[1][1]}, {&pr[1][2], &pr[1][3]}};
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                    const float x0 = *src[r4][0], x1 = *src[r4][1];
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
                    const float2 hf = __bfloat1622float2(hi);
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
                    memcpy(&pa[r4], &hi, 4);
                    memcpy(&pb[r4], &lo, 4);
                }
            }
            if (__any_sync(kFull, alpha_lo != 1.f || alpha_hi != 1.f)) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    o[j][0] *= alpha_lo;
                    o[j][1] *= alpha_lo;
                    if (ROWS16) {
                        o[j][2] *= alpha_hi;
                        o[j][3] *= alpha_hi;
                    }
                }
            }

            // O += P V (k = 16 tokens, n = head_dim in tiles of 8).
            {
                const int mi = lane >> 3;
                const int r = (lane & 7) + ((mi & 1) << 3);
#pragma unroll
                for (int jj = 0; jj < KT; ++jj) {
                    const int ch = 2 * jj + (mi >> 1);
                    const uint32_t addr =
                        Vs + (ch >> 3) * HALF_BYTES + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(addr, b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * jj], pa, b0, b1);
                    mma_bf16_16816(o[2 * jj + 1], pa, b2, b3);
                    mma_bf16_16816(o[2 * jj], pb, b0, b1);
                    mma_bf16_16816(o[2 * jj + 1], pb, b2, b3);
                }
            }
            __syncwarp();
            if (k + NSTAGE < my_n) issue(k + NSTAGE);
        }

        // Epilogue: publish this warp's state in its (now idle) stage buffers.
        l_lo += __shfl_xor_sync(kFull, l_lo, 1);
        l_lo += __shfl_xor_sync(kFull, l_lo, 2);
        if (ROWS16) {
            l_hi += __shfl_xor_sync(kFull, l_hi, 1);
            l_hi += __shfl_xor_sync(kFull, l_hi, 2);
        }
        {
            float *eo = reinterpret_cast<float *>(wbuf);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                *reinterpret_cast<float2 *>(eo + g * LD + 8 * j + 2 * t) = make_float2(o[j][0], o[j][1]);
                *reinterpret_cast<float2 *>(eo + (g + 8) * LD + 8 * j + 2 * t) =
                    ROWS16 ? make_float2(o[j][2], o[j][3]) : make_float2(0.f, 0.f);
            }
            if (t == 0) {
                eo[16 * LD + g] = m_lo;
                eo[16 * LD + 16 + g] = l_lo;
                eo[16 * LD + g + 8] = ROWS16 ? m_hi : -INFINITY;
                eo[16 * LD + 16 + g + 8] = ROWS16 ? l_hi : 0.f;
            }
        }
        if (threadIdx.x == 0) s_next[nb] = dynamic ? ahead : item + gridDim.x;
        __syncthreads();
        merge_and_store<__nv_bfloat16, HD>(smem, WARP_BYTES, p, it.seq, it.part, it.qh0, it.rows,
                                           it.single);
        fence_proxy_async_smem();
        __syncthreads();
        item = s_next[nb];
        nb ^= 1;
        if (dynamic && threadIdx.x == 0) ahead = gridDim.x + next_handout(p.work_ctr);
    }
    // No more items for this CTA: the merge launch may start taking its place
    // (it waits for this grid to finish before reading any partial).
    griddep_launch_dependents();
    if (dynamic && threadIdx.x == 0) finish_handouts(p.work_ctr);

    // A wait gave up: let copies still in flight land before the CTA exits.
    if (failed && lane == 0) {
        for (uint32_t gi = n_done; gi < n_issued; ++gi)
            mbar_wait_bounded(bar_s + 8 * (gi % NSTAGE), (gi / NSTAGE) & 1u);
    }
}

// ------------------------------------------------------- split-K reduce ---
// out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p, M = max_p m_p, for
// every (sequence, query head) whose context spans more than one partition.
// One CTA per (query head, sequence): the threads first take M over all
// partitions, then each warp sums a strided subset of the partitions (lanes own
// 4 consecutive head_dim values) and the warps' sums are added in shared memory.
template <typename OutT, int HD, int kReduceWarps>
__global__ void __launch_bounds__(kReduceWarps * 32) decode_reduce_kernel(const DecodeParams p) {
    // A following pass may be scheduled as soon as every merge CTA is running
    // (it waits for this grid before reading anything).
    griddep_launch_dependents();
    griddep_wait();   // the partition pass (launched before, programmatically) is done
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qh = blockIdx.x;
    // Newest partials first when they do not all fit in L2: the partition pass
    // writes them in sequence order, so the last sequences' are still in L2.
    const int seq = p.reduce_newest_first ? p.num_seqs - 1 - static_cast<int>(blockIdx.y)
                                          : static_cast<int>(blockIdx.y);
    const int n = seq_len(p, seq);
    if (n <= p.partition_size) return;
    const int np = (n + p.partition_size - 1) / p.partition_size;
    const long long base = (long long)seq * p.max_parts * p.num_q_heads + qh;
    const long long stride = p.num_q_heads;
    __shared__ float s_max[kReduceWarps];
    __shared__ float s_l[kReduceWarps];
    __shared__ float4 s_acc[kReduceWarps][HD / 4];
    const bool active = lane < HD / 4;

    // Staged variant (4-warp CTAs, at most kReduceMaxPartsSmall partitions):
    // every partial of the row is copied into shared memory at once (cp.async,
    // no registers held), so the row costs one round trip however many
    // partitions it has.  Otherwise (8 warps, long rows) the first kHeadParts
    // partitions of each warp are copied the same way while the maximum is
    // taken, and the rest are read as they are summed: rows of up to
    // 8 x kHeadParts partitions also cost one round trip.
    constexpr bool kStaged = kReduceWarps == 4;
    constexpr int kHeadParts = kStaged ? 1 : 4;
    extern __shared__ float4 s_stage[];            // [max_parts][HD / 4] accumulators, then [max_parts] (m, l)
    float2 *s_ml = reinterpret_cast<float2 *>(s_stage + (kStaged ? p.max_parts * (HD / 4) : 0));
    __shared__ float4 s_head[kStaged ? 1 : kHeadParts * kReduceWarps][HD / 4];
    if constexpr (kStaged) {
        if (active)
            for (int i = warp; i < np; i += kReduceWarps)
                cp_async_16(smem_addr(s_stage + i * (HD / 4) + lane), p.part_acc + (base + i * stride) * HD + lane * 4);
        for (int i = threadIdx.x; i < np; i += blockDim.x)
            cp_async_8(smem_addr(s_ml + i), p.part_ml + (base + i * stride) * 2);
        cp_async_wait_all();
        __syncthreads();
    } else {
        if (active)
#pragma unroll
            for (int j = 0; j < kHeadParts; ++j) {
                const int i = warp + j * kReduceWarps;
                if (i < np)
                    cp_async_16(smem_addr(&s_head[i][lane]), p.part_acc + (base + i * stride) * HD + lane * 4);
            }
        cp_async_commit();
    }
    auto ml_of = [&](int i) -> float2 {
        if constexpr (kStaged) return s_ml[i];
        return *reinterpret_cast<const float2 *>(p.part_ml + (base + i * stride) * 2);
    };

    float M = -INFINITY;
    for (int i = threadIdx.x; i < np; i += blockDim.x) M = fmaxf(M, ml_of(i).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    if (lane == 0) s_max[warp] = M;
    __syncthreads();
    M = s_max[0];
#pragma unroll
    for (int w = 1; w < kReduceWarps; ++w) M = fmaxf(M, s_max[w]);

    if constexpr (!kStaged) cp_async_wait_group<0>();   // this lane's head partials have landed

    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int i = warp; i < np; i += kReduceWarps) {
        const float2 ml = ml_of(i);
        const float f = exp2f(ml.x - M);
        L += f * ml.y;
        if (active) {
            float4 v;
            if constexpr (kStaged)
                v = s_stage[i * (HD / 4) + lane];
            else if (i < kHeadParts * kReduceWarps)
                v = s_head[i][lane];                   // copied by this lane, ordered by its own wait
            else
                v = *reinterpret_cast<const float4 *>(p.part_acc + (base + i * stride) * HD + lane * 4);
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
        }
    }
    if (active) s_acc[warp][lane] = acc;
    if (lane == 0) s_l[warp] = L;
    __syncthreads();
    if (warp == 0 && active) {
        float Lt = 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kReduceWarps; ++w) {
            Lt += s_l[w];
            const float4 v = s_acc[w][lane];
            a.x += v.x;
            a.y += v.y;
            a.z += v.z;
            a.w += v.w;
        }
        const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
        OutT *o = static_cast<OutT *>(p.out) + ((long long)seq * p.num_q_heads + qh) * HD + lane * 4;
        store4(o, make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv));
    }
}

}  // namespace pa

// ================================================================ host ===
namespace {

using pa::DecodeParams;

using namespace pa::host;

template <int HD, bool ROWS16>
int launch_bf16(const DecodeParams &p, const void *k_cache, const void *v_cache, long long items,
                int dev, cudaStream_t st) {
    constexpr int NS = pa::bf16_stages<HD>();
    constexpr int STAGE = 2 * (HD / 64) * pa::kChunk * 128;
    constexpr int SMEM = pa::kWarps * NS * STAGE + pa::kWarps * NS * 8 + 1024;
    static KernelSlot slot;
    auto kernel = pa::decode_bf16_kernel<HD, NS, ROWS16>;
    const int occ = ensure_kernel(kernel, slot, SMEM, dev);
    if (occ == 0) return pa_fail(PA_ERR_CUDA, "pa_decode: cannot configure the bf16 kernel");
    CUtensorMap mk, mv;
    if (!make_map(&mk, k_cache, p.total_rows, HD) || !make_map(&mv, v_cache, p.total_rows, HD))
        return pa_fail(PA_ERR_CUDA, "pa_decode: cuTensorMapEncodeTiled failed");
    const long long cap = static_cast<long long>(sm_count(dev)) * occ;
    const int grid = static_cast<int>(items < cap ? items : cap);
    const cudaError_t e = launch_dependent(kernel, grid, pa::kWarps * 32, SMEM, st, mk, mv, p);
    if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, cudaGetErrorString(e));
    return PA_OK;
}

// The merge is launched as a programmatic dependent of the partition pass: its
// CTAs may become resident while the pass's last CTAs finish, and wait in
// griddep_wait() until the pass is complete.  After any other kind of
// predecessor it simply starts when that one has finished.
// Warps per merge CTA: 4 while no sequence has more than 64 partitions -- a
// row's partials are then staged in shared memory in one round trip (at most
// 64 x (4 * head_dim + 8) bytes) -- else 8 (long sequences spread their
// partitions over more warps, read as they are summed).
constexpr int kReduceMaxPartsSmall = 64;

template <typename OutT, int HD>
cudaError_t launch_reduce(const DecodeParams &p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    const bool small = p.max_parts <= kReduceMaxPartsSmall;
    cfg.gridDim = dim3(p.num_q_heads, p.num_seqs);
    cfg.blockDim = dim3((small ? 4 : 8) * 32);
    cfg.dynamicSmemBytes = small ? static_cast<size_t>(p.max_parts) * (HD * 4 + 8) : 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return small ? cudaLaunchKernelEx(&cfg, pa::decode_reduce_kernel<OutT, HD, 4>, p)
                 : cudaLaunchKernelEx(&cfg, pa::decode_reduce_kernel<OutT, HD, 8>, p);
}

inline bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace layout: [work counter, 8 bytes, padded to 256] [partial (max, sum)]
// [partial accumulators].  The counter sits at offset 0 whatever the sizes, so
// a workspace reused for other sizes keeps a valid (zero) counter.
constexpr size_t kWorkspaceHeader = 256;

int effective_partition(int partition_size) { return partition_size == 0 ? 512 : partition_size; }

}  // namespace

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                           int max_context_len, int partition_size) {
    const int P = effective_partition(partition_size);
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len <= 0 || P <= 0) return 0;
    const long long max_parts = (static_cast<long long>(max_context_len) + P - 1) / P;
    if (max_parts <= 1) return 0;
    const size_t rows = static_cast<size_t>(num_seqs) * max_parts * num_q_heads;
    return kWorkspaceHeader + align256(rows * 2 * sizeof(float)) + align256(rows * head_dim * sizeof(float));
}

namespace {

// Argument checks shared by pa_decode and pa_decode_noalloc (everything but
// the workspace), so both entry points give the same code for the same
// mistake.  Called with num_seqs > 0.
int check_decode_args(const void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, const pa_decode_args *a) {
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: null tensor pointer");
    if (a->dtype != PA_F32 && a->dtype != PA_BF16) return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: bad dtype");
    if (a->phase < PA_PHASE_ALL || a->phase > PA_PHASE_REDUCE) return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: bad phase");
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: num_q_heads must be a positive multiple of num_kv_heads");
    if (head_dim != 64 && head_dim != 128) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: head_dim must be 64 or 128");
    if (block_size != 16 && block_size != 32) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: block_size must be 16 or 32");
    if (a->num_blocks <= 0 || a->max_blocks_per_seq <= 0 || a->max_context_len < 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: bad num_blocks, max_blocks_per_seq or max_context_len");
    const int P = effective_partition(a->partition_size);
    if (P < 16 || P > 4096 || P % 16 != 0)
        return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: partition_size must be a multiple of 16 in [16, 4096]");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: out, q and caches must be 16-byte aligned");
    const bool fused = a->k_new || a->v_new || a->slot_mapping;
    if (fused && (!a->k_new || !a->v_new || !a->slot_mapping))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: k_new, v_new and slot_mapping go together");
    if (fused && (!aligned16(a->k_new) || !aligned16(a->v_new) ||
                  (reinterpret_cast<uintptr_t>(a->slot_mapping) & 7u)))
        return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: k_new/v_new must be 16-byte and slot_mapping 8-byte aligned");
    const long long total_rows = static_cast<long long>(a->num_blocks) * num_kv_heads * block_size;
    if (total_rows >= INT_MAX) return pa_fail(PA_ERR_UNSUPPORTED, "pa_decode: cache has 2^31 or more rows");
    return PA_OK;
}

// Tokens a sequence can hold: max_context_len, bounded by the table's width.
int context_cap(const pa_decode_args *a, int block_size) {
    const long long table_cap = static_cast<long long>(a->max_blocks_per_seq) * block_size;
    return static_cast<int>(a->max_context_len < table_cap ? a->max_context_len : table_cap);
}

}  // namespace

extern "C" int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, float scale,
                         const pa_decode_args *a) {
    PaTraceRange trace("pa_decode");
    if (!a) return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: args is NULL");
    if (a->num_seqs < 0) return pa_fail(PA_ERR_INVALID_ARG, "pa_decode: num_seqs < 0");
    if (a->num_seqs == 0) return PA_OK;
    const int arc = check_decode_args(out, q, k_cache, v_cache, block_tables, context_lens, num_q_heads,
                                      num_kv_heads, head_dim, block_size, a);
    if (arc != PA_OK) return arc;
    const int P = effective_partition(a->partition_size);
    const long long total_rows = static_cast<long long>(a->num_blocks) * num_kv_heads * block_size;
    const int ctx_cap = context_cap(a, block_size);
    const int max_parts = ctx_cap <= P ? 1 : static_cast<int>((static_cast<long long>(ctx_cap) + P - 1) / P);
    DecodeParams p{};
    if (max_parts > 1) {
        const size_t need = pa_decode_workspace_size(a->num_seqs, num_q_heads, head_dim, ctx_cap, P);
        if (!a->workspace || a->workspace_bytes < need || !aligned16(a->workspace))
            return pa_fail(PA_ERR_WORKSPACE, "pa_decode: workspace missing, unaligned or smaller than pa_decode_workspace_size()");
        const size_t rows = static_cast<size_t>(a->num_seqs) * max_parts * num_q_heads;
        char *ws = static_cast<char *>(a->workspace);
        p.work_ctr = reinterpret_cast<unsigned long long *>(ws);
        p.part_ml = reinterpret_cast<float *>(ws + kWorkspaceHeader);
        p.part_acc = reinterpret_cast<float *>(ws + kWorkspaceHeader + align256(rows * 2 * sizeof(float)));
    }
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.status = a->dev_status;
    p.k_new = a->k_new;
    p.v_new = a->v_new;
    p.slot_mapping = a->slot_mapping;
    p.k_cache_w = const_cast<void *>(k_cache);
    p.v_cache_w = const_cast<void *>(v_cache);
    p.num_seqs = a->num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_q_heads / num_kv_heads;
    p.block_size = block_size;
    p.num_blocks = a->num_blocks;
    p.max_blocks_per_seq = a->max_blocks_per_seq;
    p.partition_size = P;
    p.max_parts = max_parts;
    p.ctx_cap = ctx_cap;
    p.total_rows = static_cast<int>(total_rows);
    p.scale_log2 = scale * 1.4426950408889634f;
    const bool use_mma = a->dtype == PA_BF16 && !a->simt;
    const int tile = use_mma ? 16 : 8;
    p.tile_rows = p.group < tile ? p.group : tile;
    p.head_tiles = (p.group + tile - 1) / tile;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return pa_fail(PA_ERR_CUDA, "pa_decode: no CUDA device");
    if (sm_count(dev) <= 0) return pa_fail(PA_ERR_CUDA, "pa_decode: cannot query the SM count");
    cudaStream_t st = static_cast<cudaStream_t>(a->stream);
    const long long items = static_cast<long long>(a->num_seqs) * max_parts * num_kv_heads * p.head_tiles;
    // Upper bound of the partial bytes a step writes; above the L2 size the
    // merge reads the newest partials first, while they are still there.
    const long long partial_bytes =
        static_cast<long long>(a->num_seqs) * max_parts * num_q_heads * (head_dim + 2) * 4;
    p.reduce_newest_first = max_parts > 1 && partial_bytes > l2_bytes(dev) ? 1 : 0;
    // The work counter holds hand-out indices in 32 bits; beyond that (never
    // reached by a cache that fits in memory) the fixed stride is used.
    if (items >= (1ll << 31)) p.work_ctr = nullptr;

    int rc = PA_OK;
    if (a->phase == PA_PHASE_REDUCE) {
        // only the merge pass below
    } else {
        if (p.work_ctr && !a->skip_counter_reset &&
            cudaMemsetAsync(p.work_ctr, 0, sizeof(unsigned long long), st) != cudaSuccess)
            return pa_fail(PA_ERR_CUDA, "pa_decode: cannot reset the work counter");
        if (use_mma) {
            const bool rows16 = p.group > 8;
            if (head_dim == 128)
                rc = rows16 ? launch_bf16<128, true>(p, k_cache, v_cache, items, dev, st)
                            : launch_bf16<128, false>(p, k_cache, v_cache, items, dev, st);
            else
                rc = rows16 ? launch_bf16<64, true>(p, k_cache, v_cache, items, dev, st)
                            : launch_bf16<64, false>(p, k_cache, v_cache, items, dev, st);
        } else {
            rc = pa::launch_simt_pass(p, k_cache, v_cache, a->dtype == PA_F32, head_dim, items, dev, st);
        }
    }
    if (rc != PA_OK) return rc;
    if (max_parts > 1 && a->phase != PA_PHASE_PARTITIONS) {
        cudaError_t le;
        if (a->dtype == PA_BF16)
            le = head_dim == 128 ? launch_reduce<__nv_bfloat16, 128>(p, st) : launch_reduce<__nv_bfloat16, 64>(p, st);
        else
            le = head_dim == 128 ? launch_reduce<float, 128>(p, st) : launch_reduce<float, 64>(p, st);
        if (le != cudaSuccess) return pa_fail(PA_ERR_CUDA, cudaGetErrorString(le));
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pa_fail(PA_ERR_CUDA, cudaGetErrorString(e));
    return PA_OK;
}

// ====================================================== no-alloc variant ===
// Some callers cannot allocate device memory for the split-K workspace: a
// plugin or host framework that owns every device allocation and hands the
// library only its input and output tensors, or a latency-critical path where
// a cudaMalloc (which may synchronise the device) is not allowed.  For them the
// entry point below runs the same decode with its scratch in a fixed array
// that lives in this library's device image.  The array is sized to
// PA_NOALLOC_WORKSPACE_BYTES and, like any __device__ variable, is held on
// every GPU that loads the library until the process exits.

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_WORKSPACE_BYTES];

namespace {

// Device address of g_noalloc_scratch per device.  In host code the symbol is
// only a host-side handle, never a device address, so it is resolved with
// cudaGetSymbolAddress once per device, with that device current.
void *g_noalloc_ptr[kMaxDevices] = {nullptr};
std::mutex g_noalloc_mutex;

int noalloc_scratch(int dev, void **ptr) {
    if (dev < 0 || dev >= kMaxDevices) return pa_fail(PA_ERR_CUDA, "pa_decode_noalloc: device index out of range");
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return pa_fail(PA_ERR_CUDA, "pa_decode_noalloc: cudaGetSymbolAddress of the static scratch failed");
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, const int32_t *context_lens, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size, float scale,
                                 const pa_decode_args *args) {
    PaTraceRange trace("pa_decode_noalloc");
    if (!args) return pa_fail(PA_ERR_INVALID_ARG, "pa_decode_noalloc: args is NULL");
    if (args->num_seqs < 0) return pa_fail(PA_ERR_INVALID_ARG, "pa_decode_noalloc: num_seqs < 0");
    if (args->num_seqs == 0) return PA_OK;
    // The same checks as pa_decode first, so that a bad size is reported as
    // such and not as a scratch too small for it.
    const int arc = check_decode_args(out, q, k_cache, v_cache, block_tables, context_lens, num_q_heads,
                                      num_kv_heads, head_dim, block_size, args);
    if (arc != PA_OK) return arc;
    const int P = effective_partition(args->partition_size);
    const int ctx_cap = context_cap(args, block_size);
    const size_t need = pa_decode_workspace_size(args->num_seqs, num_q_heads, head_dim, ctx_cap, P);
    if (need > PA_NOALLOC_WORKSPACE_BYTES)
        return pa_fail(PA_ERR_WORKSPACE,
                       "pa_decode_noalloc: these sizes need more split-K scratch than the library's fixed "
                       "PA_NOALLOC_WORKSPACE_BYTES; use pa_decode with a caller workspace");
    pa_decode_args a = *args;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    if (need > 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return pa_fail(PA_ERR_CUDA, "pa_decode_noalloc: no CUDA device");
        void *scratch = nullptr;
        int rc = noalloc_scratch(dev, &scratch);
        if (rc != PA_OK) return rc;
        a.workspace = scratch;
        a.workspace_bytes = PA_NOALLOC_WORKSPACE_BYTES;
    }
    return pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, &a);
}
