// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>

#include "pa.h"

// Thread-local error text for pa_last_error_string().
void pa_set_error(const char *msg);
int pa_fail(int code, const char *msg);

#ifdef __CUDACC__
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

// Names the enclosing API call as an NVTX range, so profiler timelines show
// which call enqueued which kernels.  Without a profiler attached the calls do
// nothing.
struct PaTraceRange {
    explicit PaTraceRange(const char *name) { nvtxRangePushA(name); }
    ~PaTraceRange() { nvtxRangePop(); }
    PaTraceRange(const PaTraceRange &) = delete;
    PaTraceRange &operator=(const PaTraceRange &) = delete;
};

namespace pa {

constexpr int kWarps = 4;        // warps per decode CTA
constexpr int kChunk = 16;       // tokens staged per pipeline step
constexpr int kEpiPad = 8;       // fp32 padding per row of the epilogue tile
constexpr unsigned kFull = 0xffffffffu;

// Everything a decode kernel needs besides the tensor maps.
struct DecodeParams {
    void *out;
    const void *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *part_ml;        // [S][max_parts][Hq][2]  (running max in log2 units, sum)
    float *part_acc;       // [S][max_parts][Hq][HD] (unnormalised)
    int32_t *status;
    unsigned long long *work_ctr;   // work items handed out so far (zeroed before each launch), or nullptr
    const void *k_new;     // fused cache write: [S][Hkv][HD] or nullptr
    const void *v_new;
    const int64_t *slot_mapping;
    void *k_cache_w;       // writable views of the caches (fused write only)
    void *v_cache_w;
    int num_seqs, num_q_heads, num_kv_heads, group, head_tiles, tile_rows;
    int block_size, num_blocks, max_blocks_per_seq;
    int partition_size, max_parts, ctx_cap;
    int total_rows;        // num_blocks * num_kv_heads * block_size (TMA row extent)
    int reduce_newest_first;   // merge pass walks sequences last to first
    float scale_log2;      // scale * log2(e)
};

// ------------------------------------------------------------------ PTX ---
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // bounded waits give up after ~2 s

// Wait for the phase with the given parity to complete, giving up after
// limit_ns so that a lost copy can never hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 255u) == 0 && global_timer_ns() - start > limit_ns) return false;
    }
}

// L2 policy under which the lines a load brings in are the first to be
// evicted: K/V rows are read once per step, so they should not push out the
// small, reused data (split-K partials, tables, q).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D tiled TMA load of box (x, y) into shared memory, completing on `bar`,
// with an L2 eviction-priority hint (a policy from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Programmatic dependent launch.  A kernel that ends with work for the next
// launch in its stream lets that launch start early with
// griddep_launch_dependents(); the dependent kernel calls griddep_wait()
// before it reads anything the first one wrote: the wait returns once the
// kernels it depends on have finished and their writes are visible.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Asynchronous global -> shared copies (LDGSTS) that hold no registers while
// in flight; cp_async_wait_all waits for this thread's copies.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed copy groups are in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A (16x16 bf16, row) * B (16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void flag_status(int32_t *status, int bits) {
    if (status) atomicOr(status, bits);
}

}  // namespace pa
#endif  // __CUDACC__
