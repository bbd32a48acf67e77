// Neural router f_theta and the hardware-aware routing decision (WhiFlash
// paper Sec. 3.3.2 and App. A "Neural Router Architecture"):
//   delta_al[b] = b2 + sum_j w2[j] * GELU(b1[j] + <W1[j, :], h_b>)
//   route[b]    = delta_al[b] > tau   (1 = autoregressive EAGLE-3 drafter)
// with h_b the bf16 hidden row rows[b] widened to fp32, exact-erf GELU, and
// dropout as the identity.
//
// One warp per hidden unit j (8 units per CTA).  W1 is not written by the
// kernel before this one in a round (the acceptance step), so each warp loads
// its W1 row into registers (d <= 2560) before waiting on that kernel: the
// weight stream overlaps it, and only the rows to route and the hidden states
// are read after the wait.  Each pass takes RB hidden rows, shared by the
// CTA's warps, and keeps RB dot products per warp.  STAGED (routing chosen
// rows after acceptance): the rows of the next pass stream into shared memory
// with asynchronous copies while this pass is computed.  Otherwise (every row
// of a small round, beside the LM head, which leaves no shared memory) they are
// read through L1.  Units are folded per CTA into w2[j] * GELU(z_j) partials,
// and the last CTA to finish sums the partials of every sequence in a fixed
// order (the result does not depend on CTA scheduling) and writes delta_al and
// route.
#include "wf_internal.cuh"

namespace wf {

constexpr int ROUTER_THREADS = ROUTER_UNITS_PER_CTA * 32;
constexpr int ROUTER_RB = 8;        // hidden rows per pass
constexpr int ROUTER_ROWS_PER_CTA = 32;   // rows one CTA routes (more rows: more CTAs along y)
constexpr int ROUTER_WREG = 20;     // float4 of a W1 row held per lane: d <= 32 * 4 * 20 = 2560
constexpr int ROUTER_LB = 2;        // column groups whose loads are issued together (divides WREG)
// At most 160 registers a thread: two router warps then fit in one SM
// sub-partition's 16K registers beside two warps of the LM-head kernel (up to
// 88 registers each), so the router really runs beside that kernel.
constexpr int ROUTER_MAX_REGS = 160;

__device__ __forceinline__ float gelu_erf(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }

__device__ __forceinline__ float dot4(const float4 w, const uint2 h, float acc) {
    acc = fmaf(w.x, __uint_as_float(h.x << 16), acc);
    acc = fmaf(w.y, __uint_as_float(h.x & 0xFFFF0000u), acc);
    acc = fmaf(w.z, __uint_as_float(h.y << 16), acc);
    return fmaf(w.w, __uint_as_float(h.y & 0xFFFF0000u), acc);
}

__device__ __forceinline__ void router_cp16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

template <bool STAGED>
__global__ void __maxnreg__(ROUTER_MAX_REGS)
    router_kernel(const uint16_t* __restrict__ hidden, const int32_t* __restrict__ rows, int B, int d, int m,
                  int P, const float* __restrict__ W1, const float* __restrict__ b1, const float* __restrict__ w2,
                  float b2, float tau, float* delta_al, int32_t* route, float* part, Control* ctrl) {
    // part: [B][gridDim.x] partial sums, zero on entry and on exit
    __shared__ float red[ROUTER_UNITS_PER_CTA][ROUTER_RB];
    __shared__ int s_last;
    extern __shared__ __align__(16) uint8_t rstage[];   // STAGED: two passes of RB rows (bf16)

    const int w = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * ROUTER_UNITS_PER_CTA + w;
    const int nblk = gridDim.x;
    const bool unit_live = j < m;
    const float4* wrow = reinterpret_cast<const float4*>(W1 + (size_t)(unit_live ? j : 0) * d);
    const int d4 = d >> 2;
    const bool in_regs = d4 <= 32 * ROUTER_WREG;

    // ---- independent of the predecessor: weights
    float4 wv[ROUTER_WREG];
#pragma unroll
    for (int u = 0; u < ROUTER_WREG; ++u) {
        const int c = lane + 32 * u;
        wv[u] = (in_regs && unit_live && c < d4) ? __ldg(wrow + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float bias1 = unit_live ? b1[j] : 0.f;
    const float wout = unit_live ? w2[j] : 0.f;

    // rows[] (a verify call's last_pos) comes from the kernel before this one.
    // Routing every row (rows == null) needs nothing from it: the kernel then
    // runs beside it and waits for it only before exiting, so that the kernel
    // after this one may rely on both.
    const bool beside = rows == nullptr;
    if (!beside) pdl_wait();
    pdl_trigger();

    // RB rows per pass; every warp reads the same hidden rows, straight from
    // L2 through L1 (no staging), so the CTA needs no dynamic shared memory
    // this CTA's rows: blockIdx.y picks a chunk of ROUTER_ROWS_PER_CTA
    const int y0 = blockIdx.y * ROUTER_ROWS_PER_CTA;
    const int y1 = min(B, y0 + ROUTER_ROWS_PER_CTA);
    auto row_of = [&](int bb) {   // hidden row of routed entry bb, or -1
        int r = rows ? rows[bb] : bb;   // no rows: route every row
        if (r < 0 || (P >= 0 && r >= P)) r = -1;
        return r;
    };
    const int chunks = d >> 3;   // 16-byte pieces of a row
    // STAGED: copies of pass b0's rows into buffer `which`
    auto stage = [&](int b0, int which) {
        const int nb = min(ROUTER_RB, y1 - b0);
        uint16_t* dst = reinterpret_cast<uint16_t*>(rstage) + (size_t)which * ROUTER_RB * d;
        for (int idx = threadIdx.x; idx < nb * chunks; idx += ROUTER_THREADS) {
            const int rb = idx / chunks, c = idx - rb * chunks;
            const int r = row_of(b0 + rb);
            if (r >= 0) router_cp16(dst + (size_t)rb * d + c * 8, hidden + (size_t)r * d + c * 8);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (STAGED && y0 < y1) stage(y0, 0);
    int pass = 0;
    for (int b0 = y0; b0 < y1; b0 += ROUTER_RB, ++pass) {
        const int nb = min(ROUTER_RB, y1 - b0);
        if constexpr (STAGED) {
            if (b0 + ROUTER_RB < y1) {
                stage(b0 + ROUTER_RB, (pass + 1) & 1);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            __syncthreads();
        }
        const uint2* hrow[ROUTER_RB];
        bool hv[ROUTER_RB];
#pragma unroll
        for (int rb = 0; rb < ROUTER_RB; ++rb) {
            const int r = rb < nb ? row_of(b0 + rb) : -1;
            hv[rb] = r >= 0;
            if (STAGED)
                hrow[rb] = reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(rstage) +
                                                          ((size_t)(pass & 1) * ROUTER_RB + rb) * d);
            else
                hrow[rb] = reinterpret_cast<const uint2*>(hidden + (size_t)(r >= 0 ? r : 0) * d);
        }
        float acc[ROUTER_RB];
#pragma unroll
        for (int rb = 0; rb < ROUTER_RB; ++rb) acc[rb] = 0.f;
        if (unit_live) {
            if (in_regs) {
                // loads of ROUTER_LB column groups x RB rows are issued together
                // before their FMAs, so a lane keeps LB * RB loads in flight
#pragma unroll
                for (int u0 = 0; u0 < ROUTER_WREG; u0 += ROUTER_LB) {
                    uint2 hx[ROUTER_LB][ROUTER_RB];
#pragma unroll
                    for (int u = 0; u < ROUTER_LB; ++u) {
                        const int c = lane + 32 * (u0 + u);
#pragma unroll
                        for (int rb = 0; rb < ROUTER_RB; ++rb)
                            hx[u][rb] = (hv[rb] && c < d4) ? (STAGED ? hrow[rb][c] : __ldg(hrow[rb] + c))
                                                           : make_uint2(0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < ROUTER_LB; ++u)
#pragma unroll
                        for (int rb = 0; rb < ROUTER_RB; ++rb) acc[rb] = dot4(wv[u0 + u], hx[u][rb], acc[rb]);
                }
            } else {
                for (int c0 = lane; c0 < d4; c0 += 32 * 4) {
                    float4 wl[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        wl[u] = c0 + 32 * u < d4 ? __ldg(wrow + c0 + 32 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int c = c0 + 32 * u;
                        if (c < d4) {
#pragma unroll
                            for (int rb = 0; rb < ROUTER_RB; ++rb)
                                if (hv[rb])
                                    acc[rb] = dot4(wl[u], STAGED ? hrow[rb][c] : __ldg(hrow[rb] + c), acc[rb]);
                        }
                    }
                }
            }
        }
        __syncthreads();   // the previous pass has read red[]
#pragma unroll
        for (int rb = 0; rb < ROUTER_RB; ++rb) {
            float v = acc[rb];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0 && rb < nb) red[w][rb] = unit_live ? wout * gelu_erf(v + bias1) : 0.f;
        }
        __syncthreads();
        if (threadIdx.x < nb) {
            float s = 0.f;
#pragma unroll
            for (int u = 0; u < ROUTER_UNITS_PER_CTA; ++u) s += red[u][threadIdx.x];
            part[(size_t)(b0 + threadIdx.x) * nblk + blockIdx.x] = s;
        }
    }

    // the last CTA to finish reduces the partials in a fixed order
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&ctrl->router_done, 1u) == (unsigned)(nblk * gridDim.y) - 1;
    __syncthreads();
    if (!s_last) {
        if (beside) pdl_wait();
        return;
    }
    __threadfence();
    // one warp per sequence: lane l sums partials l, l+32, ... (independent
    // loads), then a fixed xor tree - the same order on every run
    for (int b = w; b < B; b += ROUTER_UNITS_PER_CTA) {
        float* pb = part + (size_t)b * nblk;
        float s = 0.f;
        for (int c = lane; c < nblk; c += 32) s += __ldcg(pb + c);
        for (int c = lane; c < nblk; c += 32) pb[c] = 0.f;  // leave the workspace zeroed
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) {
            const int r = rows ? rows[b] : b;
            if (r < 0 || (P >= 0 && r >= P)) {
                if (delta_al) delta_al[b] = __int_as_float(0x7fc00000);
                if (route) route[b] = -1;
                record_error(ctrl, WF_ERR_BAD_DATA, (uint32_t)b);
            } else {
                s += b2;
                if (delta_al) delta_al[b] = s;
                if (route) route[b] = s > tau ? 1 : 0;
            }
        }
    }
    if (threadIdx.x == 0) ctrl->router_done = 0;
    if (beside) pdl_wait();
}

wf_status launch_router(const uint16_t* hidden, const int32_t* rows, int B, int d, int m, int P, const float* W1,
                        const float* b1, const float* w2, float b2, float tau, float* delta_al, int32_t* route,
                        void* ws, size_t part_off, cudaStream_t s) {
    if (B == 0) return WF_OK;
    Control* ctrl = reinterpret_cast<Control*>(ws);
    float* part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + part_off);
    const dim3 grid(cdiv(m, ROUTER_UNITS_PER_CTA), cdiv(B, ROUTER_ROWS_PER_CTA));
    if (rows == nullptr || d > 32 * 4 * ROUTER_WREG)
        return launch(router_kernel<false>, grid, dim3(ROUTER_THREADS), 0, s, hidden, rows, B, d, m, P, W1, b1, w2,
                      b2, tau, delta_al, route, part, ctrl);
    // chosen rows after acceptance: rows staged in shared memory, two passes in flight
    const size_t smem = (size_t)2 * ROUTER_RB * d * 2;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WF_ERR_CUDA;
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(router_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 2 * ROUTER_RB * 32 * 4 * ROUTER_WREG * 2) != cudaSuccess)
            return WF_ERR_CUDA;
        attr_set[dev] = true;
    }
    return launch(router_kernel<true>, grid, dim3(ROUTER_THREADS), smem, s, hidden, rows, B, d, m, P, W1, b1, w2,
                  b2, tau, delta_al, route, part, ctrl);
}

}  // namespace wf

namespace wf {

// Copy hidden[rows[b]] to out[b] (16-byte chunks) for an entropy sweep over
// selected rows; a row outside [0, P) is zero-filled and flagged.
__global__ void __launch_bounds__(128)
    gather_rows_kernel(const uint16_t* __restrict__ hidden, int P, int d, const int32_t* __restrict__ rows,
                       uint16_t* __restrict__ out, Control* ctrl) {
    pdl_wait();   // rows may be the previous kernel's last_pos
    pdl_trigger();
    const int b = blockIdx.x;
    const int r = rows[b];
    const bool bad = r < 0 || r >= P;
    if (bad && threadIdx.x == 0) record_error(ctrl, WF_ERR_BAD_DATA, (uint32_t)b);
    const int chunks = d >> 3;
    const uint4* src = reinterpret_cast<const uint4*>(hidden + (size_t)(bad ? 0 : r) * d);
    uint4* dst = reinterpret_cast<uint4*>(out + (size_t)b * d);
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) dst[c] = bad ? make_uint4(0, 0, 0, 0) : src[c];
}

wf_status launch_gather_rows(const uint16_t* hidden, int P, int d, const int32_t* rows, int B, uint16_t* out,
                             void* ws, cudaStream_t s) {
    return launch(gather_rows_kernel, dim3(B), dim3(128), 0, s, hidden, P, d, rows, out,
                  reinterpret_cast<Control*>(ws));
}

}  // namespace wf
