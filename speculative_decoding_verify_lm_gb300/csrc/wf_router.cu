// Neural router f_theta and the hardware-aware routing decision (WhiFlash
// paper Sec. 3.3.2 and App. A "Neural Router Architecture"):
//   delta_al[b] = b2 + sum_j w2[j] * GELU(b1[j] + <W1[j, :], h_b>)
//   route[b]    = delta_al[b] > tau   (1 = autoregressive EAGLE-3 drafter)
// with h_b the bf16 hidden row rows[b] widened to fp32, exact-erf GELU, and
// dropout as the identity.
//
// Three kernels compute it.
//
// router_kernel routes every row of a small round beside the LM head: one
// warp per hidden unit j (8 units per CTA), the W1 row held in registers
// (d <= 2560) and loaded before the dependency wait, RB hidden rows per pass
// read through L1 (no shared memory, so its CTAs fit beside the LM-head CTAs).
// Units are folded per CTA into w2[j] * GELU(z_j) partials, and the last CTA
// to finish sums them per row in a fixed order and writes delta_al and route.
//
// It also routes up to 8 chosen rows after acceptance (one pass of rows).
//
// router_gemm_kernel + router_finish_kernel route more chosen rows after
// acceptance: Z = H W1^T as a tiled fp32 GEMM on the CUDA cores (tiles of 128
// rows x 128 units, an 8 x 8 register micro-tile per thread, bf16 rows widened
// as they are staged in shared memory, K split so the CTAs fill the SMs once),
// then one CTA per row adds the K splits in order, applies b1, GELU and w2,
// sums over units in a fixed order and takes the decision.
#include "wf_internal.cuh"

namespace wf {

constexpr int ROUTER_THREADS = ROUTER_UNITS_PER_CTA * 32;
constexpr int ROUTER_RB = 8;        // hidden rows per pass
constexpr int ROUTER_ROWS_PER_CTA = 32;   // rows one CTA routes (more rows: more CTAs along y)
constexpr int ROUTER_WREG = 20;     // float4 of a W1 row held per lane: d <= 32 * 4 * 20 = 2560
constexpr int ROUTER_LB = 2;        // column groups whose loads are issued together (divides WREG)
// At most 160 registers a thread: two router warps then fit in one SM
// sub-partition's 16K registers beside two warps of the LM-head kernel (at
// most 96 registers each), so the router really runs beside that kernel.
constexpr int ROUTER_MAX_REGS = 160;

__device__ __forceinline__ float gelu_erf(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }

__device__ __forceinline__ float dot4(const float4 w, const uint2 h, float acc) {
    acc = fmaf(w.x, __uint_as_float(h.x << 16), acc);
    acc = fmaf(w.y, __uint_as_float(h.x & 0xFFFF0000u), acc);
    acc = fmaf(w.z, __uint_as_float(h.y << 16), acc);
    return fmaf(w.w, __uint_as_float(h.y & 0xFFFF0000u), acc);
}

__global__ void __maxnreg__(ROUTER_MAX_REGS)
    router_kernel(const uint16_t* __restrict__ hidden, const int32_t* __restrict__ rows, int B, int d, int m,
                  int P, const float* __restrict__ W1, const float* __restrict__ b1, const float* __restrict__ w2,
                  float b2, float tau, float* delta_al, int32_t* route, float* part, Control* ctrl) {
    // part: [B][gridDim.x] partial sums, zero on entry and on exit
    __shared__ float red[ROUTER_UNITS_PER_CTA][ROUTER_RB];
    __shared__ int s_last;

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
    for (int b0 = y0; b0 < y1; b0 += ROUTER_RB) {
        const int nb = min(ROUTER_RB, y1 - b0);
        const uint2* hrow[ROUTER_RB];
        bool hv[ROUTER_RB];
#pragma unroll
        for (int rb = 0; rb < ROUTER_RB; ++rb) {
            const int r = rb < nb ? row_of(b0 + rb) : -1;
            hv[rb] = r >= 0;
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
                            hx[u][rb] = (hv[rb] && c < d4) ? __ldg(hrow[rb] + c) : make_uint2(0u, 0u);
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
                                if (hv[rb]) acc[rb] = dot4(wl[u], __ldg(hrow[rb] + c), acc[rb]);
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

// ------------------------------------------------------------------ tiled router (chosen rows)
constexpr int RG_TB = 128;      // rows per tile
constexpr int RG_TU = 128;      // units per tile
constexpr int RG_KC = 8;        // K per shared-memory stage
constexpr int RG_THREADS = 256; // 16 x 16 threads, 8 x 8 outputs each
constexpr int RG_PD = 4;        // stages whose global loads are in flight (registers)

// Zp[ks][b][j] = sum over this split's K range of h_b[k] * W1[j, k].  Thread
// (ty, tx) = (tid / 16, tid % 16) owns rows {4ty + i, 64 + 4ty + i} and units
// {4tx + j, 64 + 4tx + j} (i, j < 4) of the tile: per K step two float4 of
// the widened rows and two of the weights feed 64 FMAs (the 4-wide halves at
// a 16-byte stride keep the weight reads free of bank conflicts; a warp reads
// two row addresses, which are broadcast).  Rows and weights are staged
// K-major in shared memory, double-buffered; RG_PD stages of each thread's
// global loads are in flight in registers.
__global__ void __launch_bounds__(RG_THREADS)
    router_gemm_kernel(const uint16_t* __restrict__ hidden, const int32_t* __restrict__ rows, int B, int d, int m,
                       int P, const float* __restrict__ W1, int kc_per, float* __restrict__ Zp) {
    __shared__ __align__(16) float Hs[2][RG_KC][RG_TB];
    __shared__ __align__(16) float Ws[2][RG_KC][RG_TU];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int u0 = blockIdx.x * RG_TU, b0 = blockIdx.y * RG_TB, ks = blockIdx.z;
    const int nkc = (d + RG_KC - 1) / RG_KC;
    const int kc0 = ks * kc_per, kc1 = min(nkc, kc0 + kc_per);
    // staging roles: row / unit tid / 2, K half (tid & 1) * 4 of a stage
    const int sr = tid >> 1, sk = (tid & 1) * 4;
    float4 wreg[RG_PD];
    uint2 hreg[RG_PD];
    const int wj = u0 + sr;
    auto load_w = [&](int kc, int slot) {   // W1 is no earlier kernel's output
        const int k = kc * RG_KC + sk;
        wreg[slot] = (kc < kc1 && wj < m && k < d) ? __ldg(reinterpret_cast<const float4*>(W1 + (size_t)wj * d + k))
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    int hsrc = -1;   // hidden row of this thread's staging row
    auto load_h = [&](int kc, int slot) {
        const int k = kc * RG_KC + sk;
        hreg[slot] = (kc < kc1 && hsrc >= 0 && k < d)
                         ? __ldg(reinterpret_cast<const uint2*>(hidden + (size_t)hsrc * d + k))
                         : make_uint2(0u, 0u);
    };
    auto store = [&](int buf, int slot) {
        const float4 wv = wreg[slot];
        Ws[buf][sk + 0][sr] = wv.x;
        Ws[buf][sk + 1][sr] = wv.y;
        Ws[buf][sk + 2][sr] = wv.z;
        Ws[buf][sk + 3][sr] = wv.w;
        const uint2 hv = hreg[slot];
        Hs[buf][sk + 0][sr] = __uint_as_float(hv.x << 16);
        Hs[buf][sk + 1][sr] = __uint_as_float(hv.x & 0xFFFF0000u);
        Hs[buf][sk + 2][sr] = __uint_as_float(hv.y << 16);
        Hs[buf][sk + 3][sr] = __uint_as_float(hv.y & 0xFFFF0000u);
    };
#pragma unroll
    for (int i = 0; i < RG_PD; ++i) load_w(kc0 + i, i);
    pdl_wait();   // rows[] is the acceptance step's output
    pdl_trigger();
    if (b0 + sr < B) {
        const int r = rows[b0 + sr];
        hsrc = (r >= 0 && (P < 0 || r < P)) ? r : -1;
    }
#pragma unroll
    for (int i = 0; i < RG_PD; ++i) load_h(kc0 + i, i);
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    if (kc0 < kc1) store(0, 0);
    __syncthreads();
    // a warp's lanes share two values of ty, so its lower rows (4 ty + i) and
    // upper rows (64 + 4 ty + i) are live or dead for the whole warp at once
    // (any live lane makes the group live): with few rows (B = 32: half the
    // warps and half of each live warp's block hold rows past B) the dead
    // groups' multiply-adds are skipped, the staging and barriers are not
    const bool lo_live = __any_sync(0xffffffffu, b0 + 4 * ty < B);
    const bool hi_live = __any_sync(0xffffffffu, b0 + 64 + 4 * ty < B);
    // stages in groups of RG_PD so that every register slot index is a constant
    for (int g0 = kc0; g0 < kc1; g0 += RG_PD) {
#pragma unroll
        for (int p = 0; p < RG_PD; ++p) {
            const int kc = g0 + p;
            if (kc >= kc1) break;
            const int buf = (kc - kc0) & 1;
            // slot p was stored for this stage: it now takes stage kc + RG_PD
            load_w(kc + RG_PD, p);
            load_h(kc + RG_PD, p);
            if (hi_live) {
#pragma unroll
                for (int k = 0; k < RG_KC; ++k) {
                    const float4 h0 = *reinterpret_cast<const float4*>(&Hs[buf][k][4 * ty]);
                    const float4 h1 = *reinterpret_cast<const float4*>(&Hs[buf][k][64 + 4 * ty]);
                    const float4 w0 = *reinterpret_cast<const float4*>(&Ws[buf][k][4 * tx]);
                    const float4 w1 = *reinterpret_cast<const float4*>(&Ws[buf][k][64 + 4 * tx]);
                    const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(hv[i], wv[j], acc[i][j]);
                }
            } else if (lo_live) {   // the upper rows are past B
#pragma unroll
                for (int k = 0; k < RG_KC; ++k) {
                    const float4 h0 = *reinterpret_cast<const float4*>(&Hs[buf][k][4 * ty]);
                    const float4 w0 = *reinterpret_cast<const float4*>(&Ws[buf][k][4 * tx]);
                    const float4 w1 = *reinterpret_cast<const float4*>(&Ws[buf][k][64 + 4 * tx]);
                    const float hv[4] = {h0.x, h0.y, h0.z, h0.w};
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(hv[i], wv[j], acc[i][j]);
                }
            }
            if (kc + 1 < kc1) {
                __syncthreads();   // the other buffer was last read a stage ago; this one is read no more
                store(buf ^ 1, (p + 1) % RG_PD);
                __syncthreads();
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int b = b0 + (i < 4 ? 4 * ty + i : 64 + 4 * ty + i - 4);
        if (b >= B) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = u0 + 64 * h + 4 * tx;
            float* z = Zp + ((size_t)ks * B + b) * m + j;
            const float* a = &acc[i][4 * h];
            if (j + 3 < m && (m & 3) == 0) {
                *reinterpret_cast<float4*>(z) = make_float4(a[0], a[1], a[2], a[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (j + q < m) z[q] = a[q];
            }
        }
    }
}

// One CTA per routed row: z_j = b1[j] + sum over the K splits (in order),
// delta = b2 + sum_j w2[j] GELU(z_j) summed in a fixed order, route = delta > tau.
// A thread owns unit j; its split partials are fetched eight at a time (all
// loads in flight together) and zeroed only after every one has been read.
constexpr int RF_THREADS = 1024;

__global__ void __launch_bounds__(RF_THREADS)
    router_finish_kernel(float* Zp, int KS, const int32_t* __restrict__ rows, int B, int m, int P,
                         const float* __restrict__ b1, const float* __restrict__ w2, float b2, float tau,
                         float* delta_al, int32_t* route, Control* ctrl) {
    __shared__ float wsum[RF_THREADS / 32];
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, tid = threadIdx.x;
    const size_t stride = (size_t)B * m;
    float t = 0.f;
    for (int j = tid; j < m; j += RF_THREADS) {
        float* zp = Zp + (size_t)b * m + j;
        float z = b1[j];
        int k = 0;
        for (; k + 8 <= KS; k += 8) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __ldcg(zp + (size_t)(k + i) * stride);
#pragma unroll
            for (int i = 0; i < 8; ++i) z += v[i];
        }
        for (; k < KS; ++k) z += __ldcg(zp + (size_t)k * stride);
        for (k = 0; k < KS; ++k) zp[(size_t)k * stride] = 0.f;   // leave the workspace zeroed
        t = fmaf(w2[j], gelu_erf(z), t);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    if ((tid & 31) == 0) wsum[tid >> 5] = t;
    __syncthreads();
    if (tid == 0) {
        float s = b2;
        for (int i = 0; i < RF_THREADS / 32; ++i) s += wsum[i];
        const int r = rows[b];
        if (r < 0 || (P >= 0 && r >= P)) {
            if (delta_al) delta_al[b] = __int_as_float(0x7fc00000);
            if (route) route[b] = -1;
            record_error(ctrl, WF_ERR_BAD_DATA, (uint32_t)b);
        } else {
            if (delta_al) delta_al[b] = s;
            if (route) route[b] = s > tau ? 1 : 0;
        }
    }
}

// K splits of the tiled router for B rows: the tiles times the splits fill
// the SMs once, a CTA an SM (the GEMM is bound by the FMA rate), within the
// workspace's partials (router_part_floats).
int router_gemm_splits(int B, int d, int m) {
    const int tiles = cdiv(B, RG_TB) * cdiv(m, RG_TU);
    const int nkc = cdiv(d, RG_KC);
    int ks = num_sms() / tiles;
    const long cap = (long)router_part_floats(B, m) / ((long)B * m);
    if (ks > cap) ks = (int)cap;
    ks = ks < 1 ? 1 : (ks > nkc ? nkc : ks);
    const int per = cdiv(nkc, ks);
    return cdiv(nkc, per);
}

wf_status launch_router(const uint16_t* hidden, const int32_t* rows, int B, int d, int m, int P, const float* W1,
                        const float* b1, const float* w2, float b2, float tau, float* delta_al, int32_t* route,
                        void* ws, size_t part_off, cudaStream_t s) {
    if (B == 0) return WF_OK;
    Control* ctrl = reinterpret_cast<Control*>(ws);
    float* part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + part_off);
    // every row of a small round beside the LM head, or a few chosen rows
    // (one pass of router_kernel): the warp-per-unit kernel, whose W1 rows
    // are in registers before the wait; more chosen rows: the tiled GEMM
    if (rows == nullptr || B <= ROUTER_RB)
        return launch(router_kernel, dim3(cdiv(m, ROUTER_UNITS_PER_CTA), cdiv(B, ROUTER_ROWS_PER_CTA)),
                      dim3(ROUTER_THREADS), 0, s, hidden, rows, B, d, m, P, W1, b1, w2, b2, tau, delta_al, route,
                      part, ctrl);
    // chosen rows: tiled GEMM with K split, then the finishing pass per row
    const int ks = router_gemm_splits(B, d, m);
    const int per = cdiv(cdiv(d, RG_KC), ks);
    const dim3 grid(cdiv(m, RG_TU), cdiv(B, RG_TB), ks);
    wf_status st = launch(router_gemm_kernel, grid, dim3(RG_THREADS), 0, s, hidden, rows, B, d, m, P, W1, per, part);
    if (st != WF_OK) return st;
    return launch(router_finish_kernel, dim3(B), dim3(RF_THREADS), 0, s, part, ks, rows, B, m, P, b1,
                  w2, b2, tau, delta_al, route, ctrl);
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
