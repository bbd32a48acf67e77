// Internal definitions shared by the library's translation units: workspace
// layout, error recording, packed argmax keys and sm_100-family PTX wrappers
// (mbarrier, TMA, tcgen05).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "wf.h"

namespace wf {

// ----------------------------------------------------------------- workspace
// [0, 256)            control block (error word, counters)   zero at rest
// [256, +8*P)         packed argmax keys, one per verified row zero at rest
// then                draft top-k candidates (no init needed)
// then                router partial sums (no init needed)
struct Control {
    uint32_t err_code;
    uint32_t err_info;
    uint32_t router_done;     // CTAs finished in the current router launch
    uint32_t gemm_done;       // CTAs finished in the current LM-head launch
    uint32_t rope_tag[2];     // catch-up: (theta bits, D + 1) of the rotary table held in the workspace
    uint32_t pad[58];
};
static_assert(sizeof(Control) == 256, "control block is 256 bytes");

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    size_t keys, cand, lsep, part, dall, ent, gath, total;
};

// Entropy statistics are kept per CTA slot; the LM-head grid never exceeds this.
constexpr int ENT_MAX_SLOTS = 160;
// Rows of one entropy sweep (at most two activation tiles).
constexpr int ENT_MAX_ROWS = 256;

// A round with at most this many verified rows runs the router on every row,
// beside the LM head while it streams its weights; the acceptance step then
// just picks the row it accepted.  Larger rounds route only the last accepted
// row of each sequence, after the acceptance step.
constexpr int ROUTE_ALL_ROWS_MAX = 128;
// The neural router runs on every row beside the LM head only for rounds this
// small: one row chunk per router CTA, all of them resident beside the LM-head
// CTAs.  Beyond it the router's sweep over all rows outlasts its benefit and it
// routes the accepted rows after acceptance instead.
constexpr int ROUTER_BESIDE_MAX_ROWS = 32;

// Merge two partial softmax states (M, S = sum e^(L-M), T = sum (L-M) e^(L-M));
// a state with S = 0 is empty and leaves the other as it is.  Written with
// selects only, so that the chains of several rows can run interleaved.
__device__ __forceinline__ void ent_merge(float& M, float& S, float& T, float m2, float s2, float t2) {
    const bool h1 = S > 0.f, h2 = s2 > 0.f;
    const float mx = h1 ? (h2 ? fmaxf(M, m2) : M) : m2;
    const float d1 = h1 ? M - mx : 0.f, d2 = h2 ? m2 - mx : 0.f;
    const float a1 = h1 ? __expf(d1) : 0.f, a2 = h2 ? __expf(d2) : 0.f;
    T = (h1 ? (T + d1 * S) * a1 : 0.f) + (h2 ? (t2 + d2 * s2) * a2 : 0.f);
    S = (h1 ? S * a1 : 0.f) + (h2 ? s2 * a2 : 0.f);
    M = mx;
}

// Optional tail of the acceptance step: the routing decision at the accepted
// row.  Either the router output of that row (computed for every row
// beforehand) is copied, or - WhiFlash-Entropy - the softmax statistics the
// LM-head sweep left per (row, CTA slot) are merged for that row alone.
struct RoutePick {
    const float* delta_all;   // [P] router output per verified row, or null
    const float4* ent;        // [P][nslots] softmax statistics (max, sum e^z, sum z e^z), or null
    int nslots;
    float tau;
    float* delta_al;          // [B]
    int32_t* route;           // [B]
    // Warp-collective (all 32 lanes, the same b and row); row < 0 marks a failed sequence.
    __device__ __forceinline__ void publish(int b, int row, int lane) const {
        if (ent) {
            constexpr int SPL = ENT_MAX_SLOTS / 32;   // slots per lane
            float4 st[SPL];
#pragma unroll
            for (int i = 0; i < SPL; ++i) {   // every load in flight before any is used
                const int sl = lane + 32 * i;
                st[i] = (row >= 0 && sl < nslots) ? __ldcg(ent + (size_t)row * nslots + sl)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float M = -INFINITY, S = 0.f, T = 0.f;
#pragma unroll
            for (int i = 0; i < SPL; ++i) ent_merge(M, S, T, st[i].x, st[i].y, st[i].z);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, M, off);
                const float s2 = __shfl_xor_sync(0xffffffffu, S, off);
                const float t2 = __shfl_xor_sync(0xffffffffu, T, off);
                ent_merge(M, S, T, m2, s2, t2);
            }
            if (lane == 0) {
                const float h = row >= 0 ? logf(S) - T / S : __int_as_float(0x7fc00000);
                delta_al[b] = h;
                route[b] = row >= 0 ? (h > tau ? 1 : 0) : -1;
            }
        } else if (delta_all && lane == 0) {
            const float v = row >= 0 ? delta_all[row] : __int_as_float(0x7fc00000);
            delta_al[b] = v;
            route[b] = row >= 0 ? (v > tau ? 1 : 0) : -1;
        }
    }
};

// tiles of the draft-head GEMM (rows x weight rows)
constexpr int BM = 128;    // activation rows per tile  (UMMA M)
constexpr int BN = 256;    // weight rows per tile      (UMMA N, largest)
constexpr int BN_MIN = 128;  // smallest weight-row tile the scheduler picks
constexpr int BK = 64;     // K elements per pipeline stage (128 bytes of bf16)
constexpr int ROUTER_UNITS_PER_CTA = 8;
// The tiled router keeps at most this many (32-row x 128-unit tile, K split)
// partial tiles of fp32 in the workspace at once (about two CTAs per SM).
constexpr int ROUTER_GEMM_SLOTS = 640;
constexpr int ROUTER_MAX_WIDTH = 65536;

inline int cdiv(long a, long b) { return (int)((a + b - 1) / b); }

// Floats of the tiled router's K-split partials ([splits][B][m]) a workspace
// holds: ROUTER_GEMM_SLOTS x 4096, and never less than one split.
inline size_t router_part_floats(int B, int m) {
    const size_t one = (size_t)(B > 0 ? B : 1) * (size_t)(m > 0 ? m : 1);
    const size_t slots = (size_t)ROUTER_GEMM_SLOTS * 4096;
    return slots > one ? slots : one;
}

// Workspace regions for a call with at most P verified rows, B sequences,
// hidden size d, router width m, draft vocabulary Vd and top-k k.
inline Layout layout(int P, int B, int d, int m, int Vd, int k) {
    P = P > 0 ? P : 0;
    B = B > 0 ? B : 0;
    const int ent_rows = B <= ENT_MAX_ROWS ? B : 0;          // rows of a gathered entropy sweep
    const int small_P = P <= ROUTE_ALL_ROWS_MAX ? P : 0;     // rows routed all at once
    Layout L;
    size_t off = sizeof(Control);
    L.keys = off;
    off = align_up(off + sizeof(uint64_t) * (size_t)(P > ent_rows ? P : ent_rows), 256);
    L.cand = off;
    L.lsep = off;
    if (Vd > 0 && k > 0) {
        size_t tiles = (size_t)cdiv(B, BM) * (size_t)cdiv(Vd, BN_MIN);
        off = align_up(off + tiles * BM * (size_t)k * sizeof(uint64_t), 256);
        // per tile and row: (max, sum of e^(logit - max)) over the tile's columns, for the log-sum-exp
        L.lsep = off;
        off = align_up(off + tiles * BM * sizeof(float2), 256);
    }
    L.part = off;
    const int routed = small_P > B ? small_P : B;
    const int mm = m > 0 ? m : 1;
    // router partials: [rows][m / 8] (beside the LM head) or [K splits][B][m]
    // of the tiled router (router_part_floats)
    const size_t beside_part = (size_t)routed * (size_t)cdiv(mm, ROUTER_UNITS_PER_CTA);
    const size_t gemm_part = router_part_floats(B, mm);
    off = align_up(off + sizeof(float) * (beside_part > gemm_part ? beside_part : gemm_part), 256);
    L.dall = off;
    off = align_up(off + sizeof(float) * (size_t)(small_P > ent_rows ? small_P : ent_rows), 256);
    L.ent = off;
    const int er = small_P > ent_rows ? small_P : ent_rows;
    off = align_up(off + sizeof(float4) * (size_t)ENT_MAX_SLOTS * (size_t)er, 256);
    L.gath = off;
    off = align_up(off + 2 * (size_t)ent_rows * (size_t)(d > 0 ? d : 0), 256);
    L.total = off;
    return L;
}

// process-wide bound on device waits (ns)
uint64_t wait_timeout_ns();
// SMs of the current device
int num_sms();
// TMA map of a [rows, cols] row-major bf16 matrix read in boxes of BK columns
// (128 bytes, 128-byte swizzle) by box_rows rows
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// One-time configuration of a call site's kernels on the current device
// (cudaFuncSetAttribute and the like), done under the site's own lock so that
// host threads making their first calls at the same time do not race on it.
// `done` holds one flag per device (devices past 64 are configured every call).
template <typename F>
inline wf_status configure_once(std::mutex& mu, bool (&done)[64], F&& configure) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WF_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && done[dev]) return WF_OK;
    if (!configure()) return WF_ERR_CUDA;
    if (dev < 64) done[dev] = true;
    return WF_OK;
}

// ----------------------------------------------------------------- launches
// Every kernel is launched with programmatic stream serialization: it may be
// scheduled while its predecessor on the stream is still running.  A kernel
// normally first waits for its predecessor (pdl_wait), then lets its own
// dependent be scheduled (pdl_trigger); before its wait it reads only inputs
// that no kernel of the round writes (weights, draft tokens, offsets), so that
// prefetch overlaps the predecessor.  The one exception, the router over all
// rows of a small round, needs nothing from its predecessor (the LM head): it
// triggers at once, computes beside it, and waits for it just before exiting -
// so its own completion still implies the LM head's.  Without the launch
// attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline wf_status launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                unsigned cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? WF_OK : WF_ERR_CUDA;
}

template <typename... KArgs, typename... Args>
inline wf_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                        Args&&... args) {
    return launch_cluster(kernel, grid, block, smem, s, 1u, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------- device helpers
__device__ __forceinline__ void record_error(Control* c, uint32_t code, uint32_t info) {
    if (atomicCAS(&c->err_code, 0u, code) == 0u) atomicExch(&c->err_info, info);
}

// Order-preserving map of an fp32 value to uint32 (larger float -> larger uint).
__device__ __forceinline__ uint32_t f32_order(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float f32_unorder(uint32_t o) {
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}
// 64-bit key: max over keys = largest logit, ties -> lowest id.  0 = empty.
__device__ __forceinline__ uint64_t pack_key(float v, uint32_t id) {
    return ((uint64_t)f32_order(v) << 32) | (uint64_t)(0xFFFFFFFFu - id);
}
__device__ __forceinline__ uint32_t key_id(uint64_t k) { return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu); }
__device__ __forceinline__ float key_val(uint64_t k) { return f32_unorder((uint32_t)(k >> 32)); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// 2^x by the PTX approximate base-2 exponential (a few ulp of fp32; results
// below the normal range flush to zero, which only drops terms under 2^-126
// of the row maximum's).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge two partial log-sum-exp states (M, S = sum e^(v - M)); S = 0 is empty.
__device__ __forceinline__ void lse_merge(float& M, float& S, float m2, float s2) {
    if (!(s2 > 0.f)) return;
    if (!(S > 0.f)) {
        M = m2;
        S = s2;
        return;
    }
    const float mx = fmaxf(M, m2);
    S = S * ex2_approx((M - mx) * LOG2E) + s2 * ex2_approx((m2 - mx) * LOG2E);
    M = mx;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// The waiting thread is suspended in hardware until the phase completes or
// about 20 us pass, so waiting warps do not take issue slots from the other
// warps (or other kernels' CTAs) on the SM.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}
// Wait until the phase with the given parity has completed, or until the
// wait has run for timeout_ns (returns false).  A non-null `abort` flag set by
// a peer role cuts the wait short.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - start > timeout_ns) return false;
    }
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// The same load issued by one CTA of a pair that computes with the paired-CTA
// MMA: the copy lands in this CTA's shared memory and its byte count is
// signalled on the mbarrier at `bar` (a shared::cluster address, here the
// first CTA's barrier, which the pair's MMA issuer waits on).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}
// shared::cluster address of the same shared-memory offset in cluster CTA `rank`
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}
// Arrive `count` times on an mbarrier of another CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// mbar_try_wait with acquire at cluster scope (a phase completed by arrivals from another CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                                  volatile int* abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t start = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - start > timeout_ns) return false;
    }
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate)
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// The paired-CTA forms (cta_group::2): the two CTAs of a cluster pair share
// one MMA of M = 256 rows - A's rows 0-127 from the first CTA's shared memory,
// 128-255 from the second's at the same offset, B's N columns split in halves
// the same way, D's rows in each CTA's own TMEM at the same address.  Both
// CTAs allocate and free their TMEM together (one warp of each); the first
// CTA issues the MMAs and commits.  Every tcgen05 instruction of such a
// kernel uses the paired form.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at shared::cluster address `bar` (this CTA's or
// the peer's) when all paired MMAs this thread issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 columns of 32-bit words from TMEM: thread t gets its lane's 32 columns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand stored as rows of
// 128 bytes with the 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B); 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1 << 16;                               // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                     // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                               // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                               // swizzle mode: 128 B
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
    return (1u << 4)                      // D format: f32
           | (1u << 7)                    // A format: bf16
           | (1u << 10)                   // B format: bf16
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

}  // namespace wf
