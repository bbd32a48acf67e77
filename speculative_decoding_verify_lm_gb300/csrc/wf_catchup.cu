// KV-only catch-up of the EAGLE-3 drafter after a switch (WhiFlash paper
// Sec. 3.4, "Lazy Catch-up" and "KV-only Prefill"; drafter geometry from the
// Qwen3-4B-EAGLE3 card, "Technical Specifications").
//
// Four launches, stream-ordered with programmatic dependent launch:
//   norm_kernel    RMSNorm of every backlog row (and a compact copy of each
//                  sequence's final row) into bf16 tensor-core operands, and
//                  the rotary frequency table
//   proj_kernel    tcgen05 GEMM  act[M, K] x W[N, K]^T  split along K over the
//                  SMs; the splits of an output tile form a thread-block
//                  cluster and sum their partial tiles over distributed shared
//                  memory in a fixed order (the result does not depend on CTA
//                  scheduling), each finishing a slice of the tile's rows:
//                    KEY    rotary embedding, bf16 rows appended to the key cache
//                    VALUE  bf16 rows appended to the value cache
//                    QUERY  rotary embedding, fp32 query of the final token
//                    OUT    residual: the final token's input plus the product
//                  One launch covers the key, value and query projections
//                  (segments of one tile space); with more than 8 sequences
//                  a second one does Wo.
//   attend_kernel  the final token's grouped-query attention over the whole
//                  cache, split along the cache rows across CTAs; the splits
//                  of each (sequence, KV head) are merged in a fixed order,
//                  inside a thread-block cluster when they fit one, else by
//                  the last CTA to arrive
//   oproj_gemv_kernel  Wo and the residual for up to 8 sequences: each CTA
//                  owns 16 output rows with the whole K, its slice of Wo in
//                  shared memory before the dependency wait (mma.sync)
//
// Every wait inside a kernel is bounded (WF_ERR_TIMEOUT, no trap).
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "wf_internal.cuh"

#define CU_TRY(x)                      \
    do {                               \
        const wf_status _st = (x);     \
        if (_st != WF_OK) return _st;  \
    } while (0)

namespace wf {

// ------------------------------------------------------------------ geometry
constexpr int PJ_STAGES = 4;
constexpr int PJ_THREADS = 192;
constexpr int PJ_A_BYTES = BM * BK * 2;           // 16 KB

constexpr int PJ_MAX_SPLIT = 8;      // K splits of one tile: the portable cluster size
constexpr int PJ_BN_CU = 192;        // widest output tile: partial, reduced and staged tiles fit the ring
constexpr int AT_MAX_CHUNKS = 64;    // cache-row splits per (sequence, KV head)
constexpr int AT_PASS_ROWS = 64;     // cache rows of one ring stage of an attention CTA
constexpr int AT_STAGES = 4;         // ring stages: three passes in flight while one is computed
constexpr int AT_SPLIT_ROWS = 256;   // smallest split of a cache worth its merge
constexpr int AT_CLUSTER_MAX = 16;   // splits merged inside one thread-block cluster (non-portable above 8)
constexpr int NORM_ROWS_PER_CTA = 4;
constexpr int NORM_REG_CHUNKS = 16;  // 16-byte pieces of a row a lane keeps in registers

enum : int { PJ_KEY = 0, PJ_VALUE = 1, PJ_QUERY = 2, PJ_OUT = 3 };

// Output tile width: whole heads, dividing both the KV width (G heads) and the
// query width (H heads), at most PJ_BN_CU columns (one head if D is wider).
inline int cu_bn(int G, int D) {
    int hp = PJ_BN_CU / D;
    if (hp < 1) hp = 1;
    while (hp > 1 && G % hp) --hp;
    return hp * D;
}

struct CuLayout {
    size_t cnt, ahat, afin, obf, q, rope, apart, total;
    int bn;
};

inline CuLayout cu_layout(int B, int N, int din, int H, int G, int D) {
    CuLayout L;
    L.bn = cu_bn(G, D);
    const int hq = H / G;
    size_t off = sizeof(Control);
    L.cnt = off;                                          // (sequence, KV head) arrivals, zero at rest
    off = align_up(off + sizeof(uint32_t) * (size_t)B * G, 256);
    L.ahat = off;
    off = align_up(off + 2 * (size_t)N * din, 256);
    L.afin = off;
    off = align_up(off + 2 * (size_t)B * din, 256);
    L.obf = off;
    off = align_up(off + 2 * (size_t)B * H * D, 256);
    L.q = off;
    off = align_up(off + 4 * (size_t)B * H * D, 256);
    L.rope = off;
    off = align_up(off + sizeof(float2) * (size_t)(D / 2), 256);
    L.apart = off;
    off = align_up(off + 4 * (size_t)B * G * AT_MAX_CHUNKS * hq * (D + 2), 256);
    L.total = off;
    return L;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// fp32 -> bf16, round to nearest even (finite inputs; NaN stays NaN)
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// Sequence of packed backlog row r: the b with bl_off[b] <= r < bl_off[b + 1].
__device__ __forceinline__ int seq_of(const int32_t* bl_off, int B, int r) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(bl_off + mid) <= r) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Rotation of the pair (x1, x2) by pos * theta^(-2i/D).  tab = theta^(-2i/D) / pi
// as a float pair hi + lo, so the angle is pi * (pos * hi + pos * lo): the
// product is split exactly (pos * hi rounded, plus its rounding error from an
// fma), the rounded part is reduced modulo 2 exactly, and sincospi takes the
// small remainder - the angle keeps ~1e-7 absolute accuracy for any position.
__device__ __forceinline__ void rope_pair(float& x1, float& x2, int pos, float2 tab) {
    const float p = (float)pos;
    const float prod = p * tab.x;
    const float err = fmaf(p, tab.x, -prod) + p * tab.y;
    const float red = prod - 2.0f * rintf(prod * 0.5f);   // exact: prod mod 2, in [-1, 1]
    float s, c;
    sincospif(red + err, &s, &c);
    const float y1 = x1 * c - x2 * s;
    const float y2 = x2 * c + x1 * s;
    x1 = y1;
    x2 = y2;
}

// ------------------------------------------------------------------ RMSNorm
// One warp per row.  Rows 0..N-1: the backlog rows (-> ahat).  Rows N..N+B-1:
// sequence b's final backlog row (-> afin), which also checks the sequence's
// offsets against its cache.  CTA 0 writes the rotary table.
__global__ void __launch_bounds__(32 * NORM_ROWS_PER_CTA)
    norm_kernel(const uint16_t* __restrict__ u, const int32_t* __restrict__ bl_off,
                const int32_t* __restrict__ cache_len, int B, int N, int din, int cap,
                const uint16_t* __restrict__ gamma, float eps, int with_final, float theta, int D,
                uint16_t* __restrict__ ahat, uint16_t* __restrict__ afin, float2* __restrict__ rope, Control* ctrl) {
    // Everything read before the dependency wait is an input of the call (the
    // backlog rows, the gains, the offsets): both row loads go out together.
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * NORM_ROWS_PER_CTA + (threadIdx.x >> 5);
    const int rows = N + (with_final ? B : 0);
    const bool active = r < rows;
    const int chunks = din >> 3;
    int src = -1, bad_b = -1;
    uint16_t* dst = nullptr;
    if (active) {
        if (r < N) {
            src = r;
            dst = ahat + (size_t)r * din;
        } else {
            const int b = r - N;
            const int n = bl_off[b + 1] - bl_off[b];
            const int L = cache_len[b];
            if (n < 1 || L < 0 || L + n > cap || bl_off[b] < 0 || bl_off[b + 1] > N)
                bad_b = b;
            else
                src = bl_off[b + 1] - 1;
            dst = afin + (size_t)b * din;
        }
    }
    const uint4* x = reinterpret_cast<const uint4*>(u + (size_t)(src < 0 ? 0 : src) * din);
    const uint4* gm = reinterpret_cast<const uint4*>(gamma);
    // rows up to 32 * NORM_REG_CHUNKS * 8 wide stay in registers (one read of the row)
    const bool in_regs = chunks <= 32 * NORM_REG_CHUNKS;
    uint4 xr[NORM_REG_CHUNKS], gr[NORM_REG_CHUNKS];
    float ss = 0.f;
    auto sumsq = [&](const uint4 v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
        }
    };
    if (src >= 0 && in_regs) {
#pragma unroll
        for (int k = 0; k < NORM_REG_CHUNKS; ++k) {
            const int c = lane + 32 * k;
            xr[k] = c < chunks ? __ldg(x + c) : make_uint4(0, 0, 0, 0);
            gr[k] = c < chunks ? __ldg(gm + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < NORM_REG_CHUNKS; ++k) sumsq(xr[k]);
    } else if (src >= 0) {
        for (int c = lane; c < chunks; c += 32) sumsq(__ldg(x + c));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rs = 1.0f / sqrtf(ss / (float)din + eps);

    // the workspace (rotary table, control block, the normalised rows) only
    // after the previous kernel on the stream is done with it
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0) {
        // the rotary table depends on (theta, D) only: it is rebuilt (in double
        // precision, slow on this GPU) only when they differ from the tagged ones
        const uint32_t tb = __float_as_uint(theta), td = (uint32_t)D + 1u;
        const bool stale = ctrl->rope_tag[0] != tb || ctrl->rope_tag[1] != td;
        if (stale && threadIdx.x < D / 2) {
            const double f = pow((double)theta, -2.0 * (double)threadIdx.x / (double)D) / 3.14159265358979323846;
            const float hi = (float)f;
            rope[threadIdx.x] = make_float2(hi, (float)(f - (double)hi));
        }
        __syncthreads();
        if (stale && threadIdx.x == 0) {
            __threadfence();
            ctrl->rope_tag[0] = tb;
            ctrl->rope_tag[1] = td;
        }
    }
    if (!active) return;
    if (src < 0) {
        if (lane == 0) record_error(ctrl, WF_ERR_BAD_DATA, (uint32_t)bad_b);
        for (int c = lane; c < chunks; c += 32) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
        return;
    }
    auto emit_g = [&](int c, const uint4 v, const uint4 gv) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w}, g[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a0 = __uint_as_float(w[j] << 16) * rs * __uint_as_float(g[j] << 16);
            const float a1 = __uint_as_float(w[j] & 0xFFFF0000u) * rs * __uint_as_float(g[j] & 0xFFFF0000u);
            o[j] = (uint32_t)f32_to_bf16(a0) | ((uint32_t)f32_to_bf16(a1) << 16);
        }
        reinterpret_cast<uint4*>(dst)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    };
    if (in_regs) {
#pragma unroll
        for (int k = 0; k < NORM_REG_CHUNKS; ++k)
            if (lane + 32 * k < chunks) emit_g(lane + 32 * k, xr[k], gr[k]);
    } else {
        for (int c = lane; c < chunks; c += 32) emit_g(c, __ldg(x + c), __ldg(gm + c));
    }
}

// ------------------------------------------------------------------ projections
struct PjSeg {
    int mode;       // PJ_KEY / PJ_VALUE / PJ_QUERY / PJ_OUT
    int a;          // activation map: 0 or 1
    int w;          // weight map: 0, 1 or 2
    int M, N;       // activation rows, output features
    int a_rows;     // rows one activation box delivers
    int tiles_n;    // output tiles along N
    int tile0;      // first tile of the segment in the launch's tile space
};

struct PjParams {
    PjSeg seg[3];
    int nseg;
    int bn, num_k, kb_per, S;   // tile width, K blocks, K blocks per split, splits (= cluster size)
    int stages, tmem_cols;      // ring stages; TMEM columns allocated (a power of two >= bn)
    uint32_t idesc;
    const int32_t* bl_off;
    const int32_t* cache_len;
    int B, N, cap, GD, HD, din;
    const float2* rope;         // [D/2]
    int D;
    uint16_t* Kc;
    uint16_t* Vc;
    float* q;                   // [B, HD]
    float* out;                 // [B, din]
    const uint16_t* u;          // backlog inputs (OUT residual)
    Control* ctrl;
    uint64_t timeout_ns;
};

// A weight box brought into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    return (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
}

__device__ __forceinline__ float4 dsmem_ld4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

struct EpiCtx {
    const PjParams& p;
    const PjSeg& g;
    int mt, r0, nrows, col0, ncols, pfs;
    uint32_t pf_local;
    const int64_t* rowdst;
    const int* rowpos;
    const float2* srope;
};

// Four columns of row rl (local row of this split's slice) starting at
// column c, summed over the S splits' partial tiles in split order (and, with
// pair_off, the same columns pair_off further on).  All of the loads are
// issued before any is used.
template <int S>
__device__ __forceinline__ void pull4(const EpiCtx& e, int rl, int c, int pair_off, float4& x, float4& x2) {
    const uint32_t off = e.pf_local + (uint32_t)(((e.r0 + rl) * e.pfs + c) * 4);
    float4 y[S], y2[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const uint32_t a = S == 1 ? off : dsmem_map(off, (uint32_t)s);
        if (S == 1) {
            y[s] = *reinterpret_cast<const float4*>(__cvta_shared_to_generic(a));
            if (pair_off) y2[s] = *reinterpret_cast<const float4*>(__cvta_shared_to_generic(a + pair_off * 4));
        } else {
            y[s] = dsmem_ld4(a);
            if (pair_off) y2[s] = dsmem_ld4(a + (uint32_t)pair_off * 4);
        }
    }
    x = y[0];
    x2 = pair_off ? y2[0] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 1; s < S; ++s) {
        x.x += y[s].x; x.y += y[s].y; x.z += y[s].z; x.w += y[s].w;
        if (pair_off) { x2.x += y2[s].x; x2.y += y2[s].y; x2.z += y2[s].z; x2.w += y2[s].w; }
    }
}

// The epilogue of one split's rows: items of 4 columns (or 4 rotation pairs),
// columns fastest, NB items per thread in flight together (NB x S x 2 vector
// loads at most 16).
template <int S>
__device__ void proj_epilogue(const EpiCtx& e) {
    constexpr int NB = 8 / S > 0 ? 8 / S : 1;
    const PjParams& p = e.p;
    const PjSeg& g = e.g;
    if (g.mode == PJ_KEY || g.mode == PJ_QUERY) {
        const int half = p.D / 2;              // a multiple of 8
        const int nq = e.ncols / 8;            // groups of 4 pairs per row
        const int items = e.nrows * nq;
        for (int base = threadIdx.x; base < items; base += NB * PJ_THREADS) {
            int rl[NB], cc[NB], ii[NB];
            float4 x1[NB], x2[NB];
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int idx = min(base + u * PJ_THREADS, items - 1);
                rl[u] = idx / nq;
                const int pi = (idx - rl[u] * nq) * 4;   // first pair of the group
                ii[u] = pi - (pi / half) * half;
                cc[u] = (pi / half) * p.D + ii[u];
                pull4<S>(e, rl[u], cc[u], half, x1[u], x2[u]);
            }
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                if (base + u * PJ_THREADS >= items) continue;
                float a1[4] = {x1[u].x, x1[u].y, x1[u].z, x1[u].w};
                float a2[4] = {x2[u].x, x2[u].y, x2[u].z, x2[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) rope_pair(a1[j], a2[j], e.rowpos[rl[u]], e.srope[ii[u] + j]);
                if (g.mode == PJ_KEY) {
                    const int64_t d = e.rowdst[rl[u]];
                    if (d >= 0) {
                        uint16_t* k1 = p.Kc + d * p.GD + e.col0 + cc[u];
                        *reinterpret_cast<uint2*>(k1) = make_uint2(pack2_bf16(a1[0], a1[1]), pack2_bf16(a1[2], a1[3]));
                        *reinterpret_cast<uint2*>(k1 + half) =
                            make_uint2(pack2_bf16(a2[0], a2[1]), pack2_bf16(a2[2], a2[3]));
                    }
                } else {
                    float* q1 = p.q + (size_t)(e.mt * BM + e.r0 + rl[u]) * p.HD + e.col0 + cc[u];
                    *reinterpret_cast<float4*>(q1) = make_float4(a1[0], a1[1], a1[2], a1[3]);
                    *reinterpret_cast<float4*>(q1 + half) = make_float4(a2[0], a2[1], a2[2], a2[3]);
                }
            }
        }
    } else {
        constexpr int NB2 = 2 * NB;
        const int nq = (e.ncols + 3) / 4;
        const int items = e.nrows * nq;
        for (int base = threadIdx.x; base < items; base += NB2 * PJ_THREADS) {
            int rl[NB2], cc[NB2];
            float4 x[NB2], unused;
#pragma unroll
            for (int u = 0; u < NB2; ++u) {
                const int idx = min(base + u * PJ_THREADS, items - 1);
                rl[u] = idx / nq;
                cc[u] = (idx - rl[u] * nq) * 4;
                pull4<S>(e, rl[u], cc[u], 0, x[u], unused);
            }
#pragma unroll
            for (int u = 0; u < NB2; ++u) {
                if (base + u * PJ_THREADS >= items) continue;
                const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                if (g.mode == PJ_VALUE) {
                    const int64_t d = e.rowdst[rl[u]];
                    if (d >= 0)   // whole heads: ncols is a multiple of 16
                        *reinterpret_cast<uint2*>(p.Vc + d * p.GD + e.col0 + cc[u]) =
                            make_uint2(pack2_bf16(xv[0], xv[1]), pack2_bf16(xv[2], xv[3]));
                } else {
                    const int f = e.rowpos[rl[u]];
                    const bool fok = f >= 0 && f < p.N;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (cc[u] + j < e.ncols) {
                            const float res = fok ? bf16_to_f32(p.u[(size_t)f * p.din + e.col0 + cc[u] + j]) : 0.f;
                            p.out[(size_t)(e.mt * BM + e.r0 + rl[u]) * p.din + e.col0 + cc[u] + j] = res + xv[j];
                        }
                }
            }
        }
    }
}

// One CTA per (output tile, K split); the S splits of a tile form one
// cluster.  Each split leaves its fp32 partial tile in its own shared memory
// (row-major, odd row pitch); after a cluster barrier, split r finishes its
// share (ceil(rows / S)) of the tile's rows, summing the S partials (in split
// order) over distributed shared memory as it goes.  Epilogue items run column
// (or rotation pair) fastest, so shared-memory reads are conflict-free and a
// warp's global stores are contiguous.  The ring holds p.stages stages of a
// 128-row activation box and a bn-row weight box; with a short ring two CTAs
// share an SM.
__global__ void __launch_bounds__(PJ_THREADS)
    proj_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                const __grid_constant__ CUtensorMap tmW2, const PjParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stages = p.stages;
    const int bstage = p.bn * BK * 2;
    uint8_t* sA = smem;
    uint8_t* sB = smem + stages * PJ_A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + stages * bstage);
    uint64_t* empty = full + stages;
    uint64_t* tfull = empty + stages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int64_t* rowdst = reinterpret_cast<int64_t*>(tmem_slot + 4);   // [BM] destination cache row, or -1
    int* rowpos = reinterpret_cast<int*>(rowdst + BM);              // [BM] position / final backlog row
    float2* srope = reinterpret_cast<float2*>(rowpos + BM);         // [D / 2] rotary table

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.S;
    const int t = blockIdx.x / S, split = blockIdx.x % S;   // split = rank in the cluster
    int si = 0;
    while (si + 1 < p.nseg && t >= p.seg[si + 1].tile0) ++si;
    const PjSeg g = p.seg[si];
    const int lt = t - g.tile0, mt = lt / g.tiles_n, nt = lt % g.tiles_n;
    const int kb0 = split * p.kb_per;
    const int kb1 = min(p.num_k, kb0 + p.kb_per);
    // the tile's rows that exist, shared out evenly: split r finishes rows [r0, r0 + nrows)
    const int tile_rows = max(0, min(BM, g.M - mt * BM));
    const int rpc = (tile_rows + S - 1) / S;
    const int r0 = min(tile_rows, split * rpc);
    const int nrows = max(0, min(rpc, tile_rows - r0));
    const CUtensorMap* mA = g.a ? &tmA1 : &tmA0;
    const CUtensorMap* mW = g.w == 0 ? &tmW0 : (g.w == 1 ? &tmW1 : &tmW2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(mA);
        tma_prefetch_desc(mW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // The weights are no earlier kernel's output: the first ring stages'
    // weight boxes are requested before waiting for the kernel that writes the
    // activations, and their activation boxes right after it.
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    const uint32_t tx = (uint32_t)(g.a_rows * BK * 2 + bstage);
    const int early = min(stages, kb1 - kb0);   // stages whose weights are requested early
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < early; ++i) {   // fresh barriers: the ring is empty
            mbar_arrive_expect_tx(&full[i], tx);
            tma_load_2d(sB + i * bstage, mW, &full[i], (kb0 + i) * BK, nt * p.bn, pol_w);
        }
        // the split's other weight boxes wait in L2 until a stage frees up
        for (int kb = kb0 + early; kb < kb1; ++kb) tma_prefetch_l2_2d(mW, kb * BK, nt * p.bn);
    }
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int i = 0; i < early; ++i)
                tma_load_2d(sA + i * PJ_A_BYTES, mA, &full[i], (kb0 + i) * BK, mt * BM, pol_a);
            int i = early;
            for (int kb = kb0 + early; kb < kb1; ++kb, ++i) {
                const int s = i % stages;
                if (!mbar_wait(&empty[s], ((i / stages) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                    *abort_flag = 1;
                    record_error(p.ctrl, WF_ERR_TIMEOUT, 0x500 + s);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], tx);
                tma_load_2d(sA + s * PJ_A_BYTES, mA, &full[s], kb * BK, mt * BM, pol_a);
                tma_load_2d(sB + s * bstage, mW, &full[s], kb * BK, nt * p.bn, pol_w);
            }
            if (*abort_flag)   // let every copy issued above land before the shared memory is reused
                for (int j = (i > stages ? i - stages : 0); j < i; ++j)
                    mbar_wait(&full[j % stages], (j / stages) & 1, p.timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int i = 0;
            for (int kb = kb0; kb < kb1; ++kb, ++i) {
                const int s = i % stages;
                if (!mbar_wait(&full[s], (i / stages) & 1, p.timeout_ns, abort_flag)) {
                    *abort_flag = 1;
                    record_error(p.ctrl, WF_ERR_TIMEOUT, 0x510 + s);
                    break;
                }
                tc_fence_after();
                const uint64_t adesc = umma_desc_sw128(smem_u32(sA + s * PJ_A_BYTES));
                const uint64_t bdesc = umma_desc_sw128(smem_u32(sB + s * bstage));
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    umma_bf16(tmem_base, adesc + 2 * kk, bdesc + 2 * kk, p.idesc, (i | kk) != 0);
                umma_commit(&empty[s]);
            }
            umma_commit(tfull);   // arrives once every MMA issued above has completed
        }
    } else {
        // ------------------------------------------------ epilogue warps: accumulator -> own partial tile
        // While the MMAs run: the rotary table and, for each row this split
        // finishes, its position and cache destination (inputs of the call).
        const int et = (int)threadIdx.x - 64;
        if ((g.mode == PJ_KEY || g.mode == PJ_QUERY) && et < p.D / 2) srope[et] = p.rope[et];
        if (et < nrows) {
            const int row = mt * BM + r0 + et;
            if (g.mode == PJ_KEY || g.mode == PJ_VALUE) {
                const int b = seq_of(p.bl_off, p.B, row);
                const int pos = p.cache_len[b] + (row - p.bl_off[b]);
                int64_t dst = -1;
                if (pos >= 0 && pos < p.cap) dst = (int64_t)b * p.cap + pos;
                else record_error(p.ctrl, WF_ERR_BAD_DATA, (uint32_t)b);
                rowdst[et] = dst;
                rowpos[et] = pos;
            } else if (g.mode == PJ_QUERY) {
                rowpos[et] = p.cache_len[row] + (p.bl_off[row + 1] - p.bl_off[row]) - 1;
            } else {
                rowpos[et] = p.bl_off[row + 1] - 1;   // the final backlog row (residual)
            }
        }
        const int q4 = warp & 3;
        const int rit = q4 * 32 + lane;
        if (!mbar_wait(tfull, 0, p.timeout_ns, abort_flag)) {
            *abort_flag = 1;
            record_error(p.ctrl, WF_ERR_TIMEOUT, 0x520);
        }
        tc_fence_after();
        if (!*abort_flag) {
            // the ring is free: every MMA (hence every copy) of this CTA has completed
            float* pf = reinterpret_cast<float*>(smem);   // [BM][bn + 4]
            const int pfs = p.bn + 4;
            const uint32_t tb = tmem_base + ((uint32_t)(q4 * 32) << 16);
            for (int c0 = 0; c0 < p.bn; c0 += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tb + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    if (c0 + j < p.bn)
                        *reinterpret_cast<uint4*>(pf + rit * pfs + c0 + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
            }
        }
        tc_fence_before();
    }
    __syncthreads();   // partial tile, row lookups and rotary table written
    if (S > 1) cluster_sync();   // every split's partial tile is in its shared memory

    // ---------------------------------------------------- epilogue of this split's rows
    // Split r finishes rows [r0, r0 + nrows) of the tile, pulling the other
    // splits' partial rows over distributed shared memory (every split's loads
    // of an item in flight together) and summing in split order.
    const int col0 = nt * p.bn;
    const int ncols = min(p.bn, g.N - col0);
    const int pfs = p.bn + 4;   // row pitch: 16-byte aligned rows for vector reads
    const uint32_t pf_local = smem_u32(smem);
    if (!*abort_flag && nrows > 0) {
        const EpiCtx e{p, g, mt, r0, nrows, col0, ncols, pfs, pf_local, rowdst, rowpos, srope};
        switch (S) {   // S <= PJ_MAX_SPLIT (host-checked)
            case 1: proj_epilogue<1>(e); break;
            case 2: proj_epilogue<2>(e); break;
            case 3: proj_epilogue<3>(e); break;
            case 4: proj_epilogue<4>(e); break;
            case 5: proj_epilogue<5>(e); break;
            case 6: proj_epilogue<6>(e); break;
            case 7: proj_epilogue<7>(e); break;
            default: proj_epilogue<8>(e); break;
        }
    }
    if (S > 1) {
        __syncthreads();
        cluster_sync();   // no CTA leaves while a peer may still read its partial tile
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ------------------------------------------------------------------ attention
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

struct AtParams {
    const float* q;            // [B, HD] rotated queries
    const uint16_t* Kc;        // [B, cap, GD]
    const uint16_t* Vc;
    const int32_t* bl_off;
    const int32_t* cache_len;
    int B, cap, G, D, hq, GD, HD, chunks;
    int cluster;               // 1: the chunks of a (sequence, KV head) form one cluster and merge over
                               // distributed shared memory; 0: through part / cnt and the last CTA
    float* part;               // [B][G][chunks][hq][D + 2]: unnormalised output, running max (log2), sum
    uint32_t* cnt;             // [B * G] arrivals, zero at rest
    uint16_t* obf;             // [B, HD] bf16 output (operand of the output projection)
    float* attn;               // [B, HD] fp32 output or null
    Control* ctrl;
    uint64_t timeout_ns;       // bound of every wait on a ring stage
};

// mma.sync m16n8k16, bf16 inputs, fp32 accumulators (row-major A, column-major B)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
}
__device__ __forceinline__ float2 dsmem_ld2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// One CTA (4 warps) per (cache-row split, KV head, sequence).  The group's hq
// <= 16 query heads form the 16 rows of an mma.sync A operand (bf16, pre-scaled
// by log2(e) / sqrt(D), padding rows zero).  The split's cache rows stream
// through a ring of AT_STAGES stages of 64 rows of K and V (asynchronous
// copies; the next three passes are in flight while one is computed, so a
// CTA keeps about 60 KB of loads outstanding) and each warp takes 16 rows of
// a pass:
//   S = Q K^T      (D/16 k-steps x 2 key tiles of 8)
//   running max / sum per head in the base-2 domain, P = exp2(S - max) as bf16
//   O += P V       (one key step of 16 x D/8 dim tiles; V fragments by ldmatrix.trans)
// Each warp keeps its own (max, sum, O) over its keys; the four are merged at
// the end.  The splits of a (sequence, KV head) are then merged in index
// order: when every such group's cluster of splits (at most AT_CLUSTER_MAX)
// can be resident at once they form one thread-block cluster, each leaves its
// partial in its own shared memory and finishes a slice of the outputs over
// distributed shared memory; otherwise partials go through global memory and
// the last CTA to arrive merges them.  The old cache
// rows of the first three passes are copied before the dependency wait.
constexpr int AT_THREADS = 128;
constexpr int AT_WARP_ROWS = 16;   // cache rows a warp takes per pass
constexpr int AT_MAX_DT = 16;      // D / 8 dim tiles: D <= 128

// DT = D / 8 dim tiles (a compile-time count: registers and unrolled loops
// for exactly the head width).
template <int DT>
__global__ void __launch_bounds__(AT_THREADS)
    attend_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const AtParams p) {
    static_assert(DT % 2 == 0 && DT >= 2 && DT <= AT_MAX_DT, "D is a multiple of 16, at most 128");
    extern __shared__ __align__(16) uint8_t smem_dyn[];
    // tensor copies land on 128-byte boundaries
    uint8_t* smem_raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
    constexpr int D = DT * 8;
    const int hq = p.hq;
    const int R = AT_PASS_ROWS;
    const int stride = D;                     // a stage's rows as the tensor copy lays them out
    const int qstride = D + 8;                // padded query rows: conflict-free fragment loads
    const size_t buf = (size_t)2 * R * stride;   // one stage: K rows then V rows
    uint16_t* Kbuf = reinterpret_cast<uint16_t*>(smem_raw);
    uint16_t* qs = Kbuf + AT_STAGES * buf;    // [16][qstride] bf16 query rows (zero padding)
    uint64_t* full = reinterpret_cast<uint64_t*>(qs + 16 * qstride);   // [AT_STAGES] stage barriers
    int* last = reinterpret_cast<int*>(full + AT_STAGES);
    float* red = reinterpret_cast<float*>(Kbuf);   // warp merge area, after the last pass

    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, cq = lane & 3;   // fragment row group, column pair
    // the split's rows follow from the call's inputs alone
    int T = p.cache_len[b] + (p.bl_off[b + 1] - p.bl_off[b]);
    T = T < 0 ? 0 : (T > p.cap ? p.cap : T);
    int Lold = p.cache_len[b];   // rows cached before this call: no kernel of the call writes them
    Lold = Lold < 0 ? 0 : (Lold > T ? T : Lold);
    const int per = (T + p.chunks - 1) / p.chunks;
    const int t0 = c * per, t1 = min(T, t0 + per);
    const int npass = t0 < t1 ? (t1 - t0 + R - 1) / R : 0;
    // A stage is one box of R cache rows x D columns of keys and one of values,
    // two tensor copies issued by one thread.  The box may run past the split
    // (those rows are masked below; past the last sequence they read as zero).
    const int gy0 = b * p.cap;   // this sequence's first row of the [B * cap, G * D] cache view
    const uint64_t pol = policy_evict_first();   // the cache is read once
    auto issue = [&](int pass) {   // thread 0
        const int which = pass % AT_STAGES;
        uint16_t* Kd = Kbuf + which * buf;
        mbar_arrive_expect_tx(&full[which], 2u * (uint32_t)R * (uint32_t)D * 2u);
        tma_load_2d(Kd, &tmK, &full[which], g * D, gy0 + t0 + pass * R, pol);
        tma_load_2d(Kd + (size_t)R * stride, &tmV, &full[which], g * D, gy0 + t0 + pass * R, pol);
    };
    bool waits_ok = true;
    auto wait_stage = [&](int pass) {
        if (!mbar_wait(&full[pass % AT_STAGES], (uint32_t)(pass / AT_STAGES) & 1u, p.timeout_ns, nullptr) &&
            waits_ok) {
            waits_ok = false;
            if (tid == 0) record_error(p.ctrl, WF_ERR_TIMEOUT, 0x600u + (uint32_t)c);
        }
    };
    constexpr int PRE = AT_STAGES - 1;
    // stages whose whole box lies in the previously cached rows (no kernel of
    // this call writes them) stream in while the kernel before this one
    // (which writes the new rows and the query) finishes; the rest after it
    int npre = 0;
    while (npre < PRE && npre < npass && t0 + (npre + 1) * R <= Lold) ++npre;
    if (tid == 0) {
        for (int i = 0; i < AT_STAGES; ++i) mbar_init(&full[i], 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        for (int i = 0; i < npre; ++i) issue(i);
    }
    // query padding rows (heads hq..15) are zero whatever the query
    for (int i = tid; i < (16 - hq) * D; i += AT_THREADS) {
        const int h = hq + i / D, e = i - (i / D) * D;
        qs[h * qstride + e] = 0;
    }
    pdl_wait();
    pdl_trigger();
    if (tid == 0)
        for (int i = npre; i < PRE && i < npass; ++i) issue(i);
    const float qscale = 1.4426950408889634f / sqrtf((float)D);
    {
        const int nq4 = hq * D / 4;   // D is a multiple of 8
        const float4* q4 = reinterpret_cast<const float4*>(p.q + (size_t)b * p.HD + (size_t)g * hq * D);
        for (int i = tid; i < nq4; i += AT_THREADS) {
            const float4 v = q4[i];
            const int h = (4 * i) / D, e = 4 * i - h * D;
            uint16_t* d = qs + h * qstride + e;
            *reinterpret_cast<uint2*>(d) = make_uint2(pack_bf16x2(v.x * qscale, v.y * qscale),
                                                      pack_bf16x2(v.z * qscale, v.w * qscale));
        }
    }
    __syncthreads();   // qs written, the stage barriers initialised

    constexpr int nks = DT / 2, ndt = DT;
    // Q fragments (A operand), one set per 16-dim k-step
    uint32_t qa[nks][4];
#pragma unroll
    for (int ks = 0; ks < nks; ++ks) {
        const int mi = lane >> 3, r = lane & 7;
        ldsm_x4(qa[ks], smem_u32(qs + ((mi & 1) * 8 + r) * qstride + ks * 16 + (mi >> 1) * 8));
    }
    float o[ndt][4];
#pragma unroll
    for (int i = 0; i < ndt; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY;   // running max of rows gq and gq + 8
    float l_lo = 0.f, l_hi = 0.f;               // this thread's share of the running sums

    for (int pass = 0; pass < npass; ++pass) {
        // refill the stage the previous pass freed: PRE passes stay in flight
        if (tid == 0 && pass + PRE < npass) issue(pass + PRE);   // the stage the previous pass freed
        wait_stage(pass);   // this pass's rows have landed
        const int p0 = t0 + pass * R;
        const uint16_t* Ks = Kbuf + (pass % AT_STAGES) * buf;
        const uint16_t* Vs = Ks + (size_t)R * stride;
        const int k0 = warp * AT_WARP_ROWS;                     // this warp's rows of the pass
        const int nvalid = min(AT_WARP_ROWS, t1 - p0 - k0);     // may be <= 0
        if (nvalid > 0) {
            // S = Q K^T over this warp's 16 rows: two 8-row key tiles
            float sc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < nks; ++ks) {
                uint32_t kb[4];   // both key tiles by one ldmatrix.x4
                const int mi = lane >> 3, r = lane & 7;
                ldsm_x4(kb, smem_u32(Ks + (size_t)(k0 + (mi >> 1) * 8 + r) * stride + ks * 16 + (mi & 1) * 8));
                mma_bf16_16816(sc[0], qa[ks], kb[0], kb[1]);
                mma_bf16_16816(sc[1], qa[ks], kb[2], kb[3]);
            }
            // mask rows past the range, then the running max / sum (rows gq, gq + 8)
            float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int key = nt * 8 + 2 * cq;
                if (key >= nvalid) sc[nt][0] = sc[nt][2] = -INFINITY;
                if (key + 1 >= nvalid) sc[nt][1] = sc[nt][3] = -INFINITY;
                mx_lo = fmaxf(mx_lo, fmaxf(sc[nt][0], sc[nt][1]));
                mx_hi = fmaxf(mx_hi, fmaxf(sc[nt][2], sc[nt][3]));
            }
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
            }
            const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
            const float a_lo = exp2f(m_lo - mn_lo), a_hi = exp2f(m_hi - mn_hi);   // 0 while the max was -inf
            m_lo = mn_lo;
            m_hi = mn_hi;
            l_lo *= a_lo;
            l_hi *= a_hi;
            if (__any_sync(0xffffffffu, a_lo != 1.f || a_hi != 1.f)) {   // a running maximum moved
#pragma unroll
                for (int i = 0; i < ndt; ++i) {
                    o[i][0] *= a_lo;
                    o[i][1] *= a_lo;
                    o[i][2] *= a_hi;
                    o[i][3] *= a_hi;
                }
            }
            uint32_t pa[4];   // P as the A operand of one 16-key step
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float p0v = exp2f(sc[nt][0] - mn_lo), p1v = exp2f(sc[nt][1] - mn_lo);
                const float p2v = exp2f(sc[nt][2] - mn_hi), p3v = exp2f(sc[nt][3] - mn_hi);
                l_lo += p0v + p1v;
                l_hi += p2v + p3v;
                pa[nt * 2 + 0] = pack_bf16x2(p0v, p1v);
                pa[nt * 2 + 1] = pack_bf16x2(p2v, p3v);
            }
            // O += P V: V fragments (keys x dims) through ldmatrix.trans; a lane
            // holds keys 2 (lane & 3) + {0, 1} (and + 8) of the step
            const int kl = 2 * cq;
            const uint32_t vmask0 = (kl < nvalid ? 0x0000FFFFu : 0u) | (kl + 1 < nvalid ? 0xFFFF0000u : 0u);
            const uint32_t vmask1 = (kl + 8 < nvalid ? 0x0000FFFFu : 0u) | (kl + 9 < nvalid ? 0xFFFF0000u : 0u);
#pragma unroll
            for (int dp = 0; dp < ndt / 2; ++dp) {   // two dim tiles per ldmatrix.x4
                uint32_t vb[4];
                const int mi = lane >> 3, r = lane & 7;
                ldsm_x4_trans(vb, smem_u32(Vs + (size_t)(k0 + (mi & 1) * 8 + r) * stride + dp * 16 + (mi >> 1) * 8));
                if (nvalid < AT_WARP_ROWS) {   // rows past the split hold any bits: P is 0 there, V must be too
                    vb[0] &= vmask0;
                    vb[2] &= vmask0;
                    vb[1] &= vmask1;
                    vb[3] &= vmask1;
                }
                mma_bf16_16816(o[2 * dp], pa, vb[0], vb[1]);
                mma_bf16_16816(o[2 * dp + 1], pa, vb[2], vb[3]);
            }
        }
        __syncthreads();   // the stage is rewritten by a later pass's copies
    }
    // sums over the four threads of each row
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
    }
    // merge the four warps: red[w][row][0..D) = O, [D] = max, [D+1] = sum
    // (4 x 16 x (D + 2) floats: within the pass buffers, 2 x 2 x 128 x (D + 8) bf16)
    const int rs = D + 2;
    float* rw = red + (size_t)warp * 16 * rs;
#pragma unroll
    for (int i = 0; i < ndt; ++i) {
        rw[gq * rs + i * 8 + 2 * cq] = o[i][0];
        rw[gq * rs + i * 8 + 2 * cq + 1] = o[i][1];
        rw[(gq + 8) * rs + i * 8 + 2 * cq] = o[i][2];
        rw[(gq + 8) * rs + i * 8 + 2 * cq + 1] = o[i][3];
    }
    if (cq == 0) {
        rw[gq * rs + D] = m_lo;
        rw[gq * rs + D + 1] = l_lo;
        rw[(gq + 8) * rs + D] = m_hi;
        rw[(gq + 8) * rs + D + 1] = l_hi;
    }
    __syncthreads();
    if (p.cluster) {
        // this split's partial stays in its own shared memory, after the warp merge area
        float* mine = red + (size_t)4 * 16 * rs;            // [hq][D + 2]
        for (int idx = tid; idx < hq * (D + 2); idx += AT_THREADS) {
            const int h = idx / (D + 2), e = idx - h * (D + 2);
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) M = fmaxf(M, red[(w * 16 + h) * rs + D]);
            float v = 0.f;
            if (e == D) {
                v = M;
            } else {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float mw = red[(w * 16 + h) * rs + D];
                    const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
                    v = fmaf(wt, red[(w * 16 + h) * rs + (e == D + 1 ? D + 1 : e)], v);
                }
            }
            mine[idx] = v;
        }
        cluster_sync();   // every split's partial is in its shared memory
        // this split finishes output pairs [c * per_c, (c + 1) * per_c): a
        // thread fetches every split's (max, sum) of its head and its two
        // values in one batch, then weighs the splits in index order
        const int CS = p.chunks;
        const uint32_t mine_s = smem_u32(mine);
        const int items = hq * (D / 2);
        const int per_c = (items + CS - 1) / CS;
        const int i1 = min(items, (c + 1) * per_c);
        for (int it = c * per_c + tid; it < i1; it += AT_THREADS) {
            const int h = it / (D / 2), e = it - h * (D / 2);
            const uint32_t av = mine_s + (uint32_t)((h * (D + 2) + 2 * e) * 4);
            const uint32_t as = mine_s + (uint32_t)((h * (D + 2) + D) * 4);   // (max, sum), adjacent
            float2 ov[AT_CLUSTER_MAX], st[AT_CLUSTER_MAX];
#pragma unroll
            for (int s2 = 0; s2 < AT_CLUSTER_MAX; ++s2)
                if (s2 < CS) {
                    ov[s2] = dsmem_ld2(dsmem_map(av, (uint32_t)s2));
                    st[s2] = dsmem_ld2(dsmem_map(as, (uint32_t)s2));
                }
            float M = -INFINITY;
#pragma unroll
            for (int s2 = 0; s2 < AT_CLUSTER_MAX; ++s2)
                if (s2 < CS) M = fmaxf(M, st[s2].x);
            float L = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < AT_CLUSTER_MAX; ++s2)
                if (s2 < CS) {
                    const float w = st[s2].x == -INFINITY ? 0.f : exp2f(st[s2].x - M);   // a split with no rows weighs 0
                    L = fmaf(w, st[s2].y, L);
                    a0 = fmaf(w, ov[s2].x, a0);
                    a1 = fmaf(w, ov[s2].y, a1);
                }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const float r0 = a0 * inv, r1 = a1 * inv;
            const size_t o2 = (size_t)b * p.HD + ((size_t)g * hq + h) * D + 2 * e;
            *reinterpret_cast<uint32_t*>(p.obf + o2) = pack_bf16x2(r0, r1);
            if (p.attn) {
                p.attn[o2] = r0;
                p.attn[o2 + 1] = r1;
            }
        }
        cluster_sync();   // no split leaves while a peer may still read its partial
        return;
    }
    float* mypart = p.part + (((size_t)b * p.G + g) * p.chunks + c) * hq * (D + 2);
    for (int idx = tid; idx < hq * (D + 2); idx += AT_THREADS) {
        const int h = idx / (D + 2), e = idx - h * (D + 2);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, red[(w * 16 + h) * rs + D]);
        float v = 0.f;
        if (e == D) {
            v = M;
        } else {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float mw = red[(w * 16 + h) * rs + D];
                const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
                v = fmaf(wt, red[(w * 16 + h) * rs + (e == D + 1 ? D + 1 : e)], v);
            }
        }
        mypart[idx] = v;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) *last = atomicAdd(&p.cnt[(size_t)b * p.G + g], 1u) == (uint32_t)(p.chunks - 1);
    __syncthreads();
    if (!*last) return;
    __threadfence();
    // merge the splits in index order: every split's (max, sum) per head into
    // shared memory (the pass buffers are free now), one weight per split and
    // head, then each output element sums the splits with independent loads
    const float* allp = p.part + ((size_t)b * p.G + g) * p.chunks * hq * (D + 2);
    // every split's partial (outputs, max, sum) of this (sequence, KV head) into
    // shared memory at once, when it fits beside the weights; else read from L2
    const size_t nf = (size_t)p.chunks * hq * (D + 2);
    const bool staged = (nf + 2 * (size_t)p.chunks * hq + hq) * 4 <= AT_STAGES * buf * 2;
    float* pm = reinterpret_cast<float*>(Kbuf);                 // [chunks][hq][D + 2] (staged)
    float* wgt = staged ? pm + nf : reinterpret_cast<float*>(Kbuf);   // [chunks][hq] split weights
    float* lsum = wgt + (size_t)p.chunks * hq;                  // [chunks][hq] split sums
    float* mtot = lsum + (size_t)p.chunks * hq;                 // [hq] 1 / merged sum
    if (staged) {
        for (size_t i = tid; i < nf / 2; i += AT_THREADS)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(pm + 2 * i)), "l"(allp + 2 * i)
                         : "memory");
        cp_async_commit();
        cp_async_wait_0();
        __syncthreads();
    }
    const float* src = staged ? pm : allp;
    for (int idx = tid; idx < p.chunks * hq; idx += AT_THREADS) {
        wgt[idx] = staged ? src[(size_t)idx * (D + 2) + D] : __ldcg(src + (size_t)idx * (D + 2) + D);
        lsum[idx] = staged ? src[(size_t)idx * (D + 2) + D + 1] : __ldcg(src + (size_t)idx * (D + 2) + D + 1);
    }
    __syncthreads();
    if (tid < hq) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < p.chunks; ++s2) M = fmaxf(M, wgt[s2 * hq + tid]);
        float L = 0.f;
        for (int s2 = 0; s2 < p.chunks; ++s2) {
            const float ms = wgt[s2 * hq + tid];
            const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);   // a split with no rows weighs 0
            wgt[s2 * hq + tid] = w;
            L = fmaf(w, lsum[s2 * hq + tid], L);
        }
        mtot[tid] = L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
    // two output pairs per thread at a time, eight splits each per step
    const int nitems = hq * D / 2;
    for (int base = tid; base < nitems; base += 2 * AT_THREADS) {
        int hh[2], ee[2];
        bool live[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int idx = base + u * AT_THREADS;
            live[u] = idx < nitems;
            const int id = live[u] ? idx : 0;
            hh[u] = id / (D / 2);
            ee[u] = id - hh[u] * (D / 2);
        }
        float a0[2] = {0.f, 0.f}, a1[2] = {0.f, 0.f};
        for (int s0 = 0; s0 < p.chunks; s0 += 8) {
            float2 ov[2][8];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float* q2 = src + ((size_t)(s0 + j) * hq + hh[u]) * (D + 2) + 2 * ee[u];
                    ov[u][j] = (s0 + j < p.chunks)
                                   ? (staged ? *reinterpret_cast<const float2*>(q2)
                                             : __ldcg(reinterpret_cast<const float2*>(q2)))
                                   : make_float2(0.f, 0.f);
                }
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (s0 + j < p.chunks) {
                        const float w = wgt[(s0 + j) * hq + hh[u]];
                        a0[u] = fmaf(w, ov[u][j].x, a0[u]);
                        a1[u] = fmaf(w, ov[u][j].y, a1[u]);
                    }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
            if (live[u]) {
                const float r0 = a0[u] * mtot[hh[u]], r1 = a1[u] * mtot[hh[u]];
                const size_t o2 = (size_t)b * p.HD + ((size_t)g * hq + hh[u]) * D + 2 * ee[u];
                *reinterpret_cast<uint32_t*>(p.obf + o2) = pack_bf16x2(r0, r1);
                if (p.attn) {
                    p.attn[o2] = r0;
                    p.attn[o2 + 1] = r1;
                }
            }
    }
    if (tid == 0) p.cnt[(size_t)b * p.G + g] = 0;
}

// ------------------------------------------------------------------ output projection, few rows
// out[b, n] = u[final row of b, n] + sum_k obf[b, k] Wo[n, k] for B <= OG_MAX_B
// rows.  CTA c owns output rows [16 c, 16 c + 16) with the whole K: its slice
// of Wo (16 consecutive rows) and the residual entries are copied into shared
// memory before the dependency wait (neither is an earlier kernel's output),
// so after it only the B attention rows are fetched, and no K split means no
// reduction between CTAs.  The product runs on mma.sync m16n8k16 (bf16
// operands, fp32 accumulators): output rows are M (one tile of 16), the B
// rows N (8, zero-padded), each of the 8 warps takes a contiguous eighth of
// the K steps and loads its B fragments straight from global memory (all in
// flight together), and the warps' partial tiles are summed in warp order.
// Weight rows are padded by 16 bytes so that ldmatrix reads are free of bank
// conflicts.  At about 87 KB of shared memory (HD = 2560) a CTA fits beside
// an attention CTA, so the whole grid is resident, and its weights in flight,
// while the attention runs.
constexpr int OG_THREADS = 256;
constexpr int OG_WARPS = OG_THREADS / 32;
constexpr int OG_MAX_B = 8;
constexpr int OG_R = 16;         // output rows a CTA owns: one 16-row tile
constexpr int OG_MAX_KPW = 24;   // K steps of 16 a warp takes: HD <= 8 x 24 x 16

struct OgParams {
    const uint16_t* Wo;   // [din, HD]
    const uint16_t* obf;  // [B, HD] attention output (bf16)
    const uint16_t* u;    // [N, din] backlog inputs (residual)
    const int32_t* bl_off;
    float* out;           // [B, din]
    int B, N, din, HD;
};

__global__ void __launch_bounds__(OG_THREADS) oproj_gemv_kernel(const OgParams p) {
    extern __shared__ __align__(16) uint8_t og_smem[];
    constexpr int R = OG_R;
    const int HD = p.HD, B = p.B;
    const int pitch = HD + 8;                                          // bf16 elements per shared row
    uint16_t* Ws = reinterpret_cast<uint16_t*>(og_smem);               // [16][pitch] weight rows
    float* res = reinterpret_cast<float*>(Ws + (size_t)R * pitch);     // [B][16] residual entries
    float* red = res + OG_MAX_B * R;                                   // [warps][16][8] partial tiles
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * R;
    const int nr = min(R, p.din - n0);
    const int cpr = HD / 8;   // 16-byte pieces of a row
    const uint16_t* wsrc = p.Wo + (size_t)n0 * HD;
    for (int i = tid; i < nr * cpr; i += OG_THREADS) {
        const int r = i / cpr, j = i - r * cpr;
        cp_async16(Ws + (size_t)r * pitch + j * 8, wsrc + (size_t)r * HD + j * 8);
    }
    cp_async_commit();
    // rows the MMAs read but no output keeps: zero, so they hold numbers
    for (int i = tid; i < (R - nr) * cpr; i += OG_THREADS) {
        const int r = nr + i / cpr, j = i - (i / cpr) * cpr;
        *reinterpret_cast<uint4*>(Ws + (size_t)r * pitch + j * 8) = make_uint4(0, 0, 0, 0);
    }
    for (int i = tid; i < B * R; i += OG_THREADS) {
        const int b = i / R, r = i - b * R;
        const int f = p.bl_off[b + 1] - 1;   // the final backlog row of sequence b
        res[i] = (r < nr && f >= 0 && f < p.N) ? bf16_to_f32(p.u[(size_t)f * p.din + n0 + r]) : 0.f;
    }
    const int nks = HD / 16;
    const int kper = (nks + OG_WARPS - 1) / OG_WARPS;
    const int k0 = warp * kper, k1 = min(nks, k0 + kper);
    const int gq = lane >> 2, cq = lane & 3;
    pdl_wait();   // obf is the attention kernel's output
    pdl_trigger();
    // B fragments of this warp's K steps: row gq of the attention output,
    // columns 16 ks + 2 cq (+1) and 16 ks + 8 + 2 cq (+1)
    uint32_t bf[OG_MAX_KPW][2];
#pragma unroll
    for (int j = 0; j < OG_MAX_KPW; ++j) {
        const int ks = k0 + j;
        const bool ok = ks < k1 && gq < B;
        const unsigned int* src = reinterpret_cast<const unsigned int*>(p.obf + (size_t)gq * HD + ks * 16 + 2 * cq);
        bf[j][0] = ok ? __ldcg(src) : 0u;
        bf[j][1] = ok ? __ldcg(src + 4) : 0u;
    }
    cp_async_wait_0();
    __syncthreads();   // the weight slice has landed
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
    for (int j = 0; j < OG_MAX_KPW; ++j) {
        const int ks = k0 + j;
        if (ks >= k1) break;
        uint32_t a[4];
        ldsm_x4(a, smem_u32(Ws + (size_t)((mi & 1) * 8 + r8) * pitch + ks * 16 + (mi >> 1) * 8));
        mma_bf16_16816(c, a, bf[j][0], bf[j][1]);
    }
    // partial tiles -> shared memory: thread holds rows gq, gq + 8 and columns 2 cq, 2 cq + 1
    float* rw = red + (size_t)warp * R * 8;
    rw[gq * 8 + 2 * cq] = c[0];
    rw[gq * 8 + 2 * cq + 1] = c[1];
    rw[(gq + 8) * 8 + 2 * cq] = c[2];
    rw[(gq + 8) * 8 + 2 * cq + 1] = c[3];
    __syncthreads();
    if (tid < R * 8) {
        const int row = tid >> 3, col = tid & 7;   // 16 rows x 8 columns, one a thread
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < OG_WARPS; ++w) v += red[(size_t)w * R * 8 + row * 8 + col];
        if (row < nr && col < B) p.out[(size_t)col * p.din + n0 + row] = res[col * R + row] + v;
    }
}

size_t catchup_oproj_gemv_smem(int HD) {
    return (size_t)OG_R * (HD + 8) * 2 + (size_t)OG_MAX_B * OG_R * 4 + (size_t)OG_WARPS * OG_R * 8 * 4;
}

// ------------------------------------------------------------------ host side
// Shared memory of a proj_kernel CTA with `stages` ring stages of tile width bn.
static size_t proj_smem(int stages, int bn) {
    return 1024 + (size_t)stages * (PJ_A_BYTES + (size_t)bn * BK * 2) + 256 + BM * 12 + 512;
}

static wf_status launch_proj(const CUtensorMap* mA, const CUtensorMap* mW, PjParams p, int tiles, cudaStream_t s) {
    static std::mutex mu;
    static bool attr_set[64] = {false};
    // Every catch-up kernel asks for the largest shared-memory carveout, so
    // that an SM need not drain to switch it when the next kernel's CTAs
    // arrive (they then start beside the previous kernel's last CTAs).
    CU_TRY(configure_once(mu, attr_set, [] {
        return cudaFuncSetAttribute(proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)proj_smem(PJ_STAGES, PJ_BN_CU)) == cudaSuccess &&
               cudaFuncSetAttribute(proj_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess;
    }));
    // A three-stage ring lets two CTAs share an SM when the tile is narrow;
    // the partial tile ([BM][bn + 4] fp32) reuses the ring and must fit in it.
    int stages = 3;
    if (2 * (proj_smem(stages, p.bn) + 1024) > 228 * 1024) stages = PJ_STAGES;
    while ((size_t)stages * (PJ_A_BYTES + (size_t)p.bn * BK * 2) < (size_t)BM * (p.bn + 4) * 4) ++stages;
    const size_t smem = proj_smem(stages, p.bn);
    const int per_sm = 2 * (smem + 1024) <= 228 * 1024 ? 2 : 1;
    p.stages = stages;
    p.tmem_cols = 32;
    while (p.tmem_cols < p.bn) p.tmem_cols *= 2;
    // split K (up to the portable cluster size): the most splits that keep
    // the CTAs at about 1.6 an SM (8/5) when two fit, one otherwise, and at
    // least two K blocks a split.  (Measured on a GB300 over S = 2..8: 1,024
    // backlog rows - 80 tiles - take S = 3, 55 us a call against 59 at S = 2
    // and 69 at S = 8; 24 tiles take S = 8; 32 tiles S = 7.)
    const int budget = per_sm == 2 ? 8 * num_sms() / 5 : num_sms();
    int S = 1;
    while (S < PJ_MAX_SPLIT && tiles * (S + 1) <= budget && 2 * (S + 1) <= p.num_k) ++S;
    p.kb_per = cdiv(p.num_k, S);
    while (S > 1 && (S - 1) * p.kb_per >= p.num_k) S /= 2;   // every split gets at least one K block
    p.kb_per = cdiv(p.num_k, S);
    p.S = S;
    return launch_cluster(proj_kernel, dim3(tiles * S), dim3(PJ_THREADS), smem, s, (unsigned)S, mA[0], mA[1],
                          mW[0], mW[1], mW[2], p);
}

static PjParams proj_params(const wf_catchup_args* a, const CuLayout& L, void* ws) {
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    PjParams p = {};
    p.bn = L.bn;
    p.idesc = umma_idesc_bf16(BM, L.bn);
    p.bl_off = a->bl_off;
    p.cache_len = a->cache_len;
    p.B = a->B;
    p.N = a->N;
    p.cap = a->cap;
    p.GD = a->G * a->D;
    p.HD = a->H * a->D;
    p.din = a->din;
    p.rope = reinterpret_cast<const float2*>(w + L.rope);
    p.D = a->D;
    p.Kc = a->Kc;
    p.Vc = a->Vc;
    p.q = reinterpret_cast<float*>(w + L.q);
    p.out = a->out;
    p.u = a->u;
    p.ctrl = reinterpret_cast<Control*>(ws);
    p.timeout_ns = wait_timeout_ns();
    return p;
}

static int add_seg(PjParams& p, int tile0, int mode, int am, int wm, int M, int N, int bn) {
    PjSeg& g = p.seg[p.nseg++];
    g.mode = mode;
    g.a = am;
    g.w = wm;
    g.M = M;
    g.N = N;
    g.a_rows = M <= BM ? (M + 7) / 8 * 8 : BM;
    g.tiles_n = cdiv(N, bn);
    g.tile0 = tile0;
    return tile0 + cdiv(M, BM) * g.tiles_n;
}

// act [rows, cols] box: the rows present (one tile) or BM
static bool act_map(CUtensorMap* m, const void* base, int rows, int cols) {
    return make_map(m, base, (uint64_t)rows, (uint64_t)cols, (uint32_t)(rows <= BM ? (rows + 7) / 8 * 8 : BM));
}

size_t catchup_attend_smem(int H, int G, int D);

using AttendFn = void (*)(CUtensorMap, CUtensorMap, AtParams);
// the attention kernel for head width D (a multiple of 16 up to 128)
static AttendFn attend_fn(int D) {
    switch (D / 8) {
        case 2: return attend_kernel<2>;
        case 4: return attend_kernel<4>;
        case 6: return attend_kernel<6>;
        case 8: return attend_kernel<8>;
        case 10: return attend_kernel<10>;
        case 12: return attend_kernel<12>;
        case 14: return attend_kernel<14>;
        case 16: return attend_kernel<16>;
        default: return nullptr;
    }
}

// [rows, cols] bf16 cache view, boxes of D columns x AT_PASS_ROWS rows laid
// out densely (no swizzle); rows past the view read as zero
static bool cache_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, int D) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)AT_PASS_ROWS};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// How many clusters of `size` attention CTAs with `smem` bytes each can be
// resident at once (one query per device, size and shared-memory size; the
// cache is shared by host threads).
static int attend_resident_clusters(int dev, int size, size_t smem, AttendFn fn) {
    struct Entry {
        int dev, size;
        size_t smem;
        AttendFn fn;
        int n;
    };
    static Entry seen[64];
    static int nseen = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < nseen; ++i)
        if (seen[i].dev == dev && seen[i].size == size && seen[i].smem == smem && seen[i].fn == fn)
            return seen[i].n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(size, 1, 1);
    cfg.blockDim = dim3(AT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = size;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    if (nseen < 64) seen[nseen++] = {dev, size, smem, fn, n};
    return n;
}

wf_status launch_catchup(const wf_catchup_args* a, void* ws, bool with_final, cudaStream_t s) {
    const CuLayout L = cu_layout(a->B, a->N, a->din, a->H, a->G, a->D);
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    Control* ctrl = reinterpret_cast<Control*>(ws);
    uint16_t* ahat = reinterpret_cast<uint16_t*>(w + L.ahat);
    uint16_t* afin = reinterpret_cast<uint16_t*>(w + L.afin);
    const int GD = a->G * a->D, HD = a->H * a->D;
    const int rows = a->N + (with_final ? a->B : 0);
    static std::mutex norm_mu;
    static bool norm_attr[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WF_ERR_CUDA;
    CU_TRY(configure_once(norm_mu, norm_attr, [] {   // see launch_proj: the largest shared-memory carveout
        return cudaFuncSetAttribute(norm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess;
    }));
    CU_TRY(launch(norm_kernel, dim3(cdiv(rows, NORM_ROWS_PER_CTA)), dim3(32 * NORM_ROWS_PER_CTA), 0, s, a->u,
                         a->bl_off, a->cache_len, a->B, a->N, a->din, a->cap, a->gamma, a->eps, (int)with_final,
                         a->theta, a->D, ahat, afin, reinterpret_cast<float2*>(w + L.rope), ctrl));
    // keys, values (and the final token's query) in one launch
    CUtensorMap mA[2], mW[3];
    if (!act_map(&mA[0], ahat, a->N, a->din) || !make_map(&mW[0], a->Wk, GD, a->din, L.bn) ||
        !make_map(&mW[1], a->Wv, GD, a->din, L.bn))
        return WF_ERR_CUDA;
    mA[1] = mA[0];
    mW[2] = mW[0];
    PjParams p = proj_params(a, L, ws);
    p.num_k = cdiv(a->din, BK);
    int tiles = add_seg(p, 0, PJ_KEY, 0, 0, a->N, GD, L.bn);
    tiles = add_seg(p, tiles, PJ_VALUE, 0, 1, a->N, GD, L.bn);
    if (with_final) {
        if (!act_map(&mA[1], afin, a->B, a->din) || !make_map(&mW[2], a->Wq, HD, a->din, L.bn)) return WF_ERR_CUDA;
        tiles = add_seg(p, tiles, PJ_QUERY, 1, 2, a->B, HD, L.bn);
    }
    CU_TRY(launch_proj(mA, mW, p, tiles, s));
    if (!with_final) return WF_OK;

    // the final token's attention over its whole cache
    AtParams ap = {};
    ap.q = reinterpret_cast<const float*>(w + L.q);
    ap.Kc = a->Kc;
    ap.Vc = a->Vc;
    ap.bl_off = a->bl_off;
    ap.cache_len = a->cache_len;
    ap.B = a->B;
    ap.cap = a->cap;
    ap.G = a->G;
    ap.D = a->D;
    ap.hq = a->H / a->G;
    ap.GD = GD;
    ap.HD = HD;
    // splits of each sequence's cache rows: about 1.25 CTAs an SM over all
    // (sequence, KV head) pairs, at most AT_CLUSTER_MAX (so that a split's
    // partials can merge on chip), and no split shorter than AT_SPLIT_ROWS of
    // the cache capacity - short splits cost more to merge than to read.
    // (Measured on a GB300, S = 2..38 a sequence: 8 x 128 onto 8,192 takes 3
    // splits, 69 us a call against 72 at 4 and 73 at 8; 1,024 onto 16,384
    // takes 16, 46 us against 48 at 38 with the global merge.)
    const int want = cdiv(5 * num_sms(), 4 * a->B * a->G);
    const int by_rows = cdiv(a->cap, AT_SPLIT_ROWS);
    int chunks = want < by_rows ? want : by_rows;
    if (chunks > AT_CLUSTER_MAX) chunks = AT_CLUSTER_MAX;
    ap.chunks = chunks < 1 ? 1 : (chunks > AT_MAX_CHUNKS ? AT_MAX_CHUNKS : chunks);
    ap.part = reinterpret_cast<float*>(w + L.apart);
    ap.cnt = reinterpret_cast<uint32_t*>(w + L.cnt);
    ap.obf = reinterpret_cast<uint16_t*>(w + L.obf);
    ap.attn = a->attn;
    ap.ctrl = ctrl;
    ap.timeout_ns = wait_timeout_ns();
    const size_t at_smem = catchup_attend_smem(a->H, a->G, a->D);
    static std::mutex at_mu;
    static bool at_attr[64] = {false};
    const AttendFn at_fn = attend_fn(a->D);
    if (!at_fn) return WF_ERR_INVALID_ARG;
    CU_TRY(configure_once(at_mu, at_attr, [] {
        for (int dt = 2; dt <= AT_MAX_DT; dt += 2) {
            const AttendFn f = attend_fn(dt * 8);
            if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess ||
                cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess ||
                cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
                return false;
        }
        return true;
    }));
    // few splits: each (sequence, KV head) is one cluster and merges on chip,
    // provided all of the clusters are resident at once (a CTA that finishes
    // early holds its slot until its cluster has merged)
    ap.cluster = ap.chunks > 1 && ap.chunks <= AT_CLUSTER_MAX &&
                         a->B * a->G <= attend_resident_clusters(dev, ap.chunks, at_smem, at_fn)
                     ? 1
                     : 0;
    CUtensorMap tmK, tmV;
    if (!cache_map(&tmK, a->Kc, (uint64_t)a->B * a->cap, GD, a->D) ||
        !cache_map(&tmV, a->Vc, (uint64_t)a->B * a->cap, GD, a->D))
        return WF_ERR_CUDA;
    CU_TRY(launch_cluster(at_fn, dim3(ap.chunks, a->G, a->B), dim3(AT_THREADS), at_smem, s,
                          ap.cluster ? (unsigned)ap.chunks : 1u, tmK, tmV, ap));

    // output projection with the residual: a GEMV for a few rows whose weight
    // slices fit in shared memory in one wave, else the tensor-core kernel
    const int og_ctas = cdiv(a->din, OG_R);
    const size_t og_smem = catchup_oproj_gemv_smem(HD);
    if (a->B <= OG_MAX_B && og_ctas <= 2 * num_sms() && HD <= OG_WARPS * OG_MAX_KPW * 16 &&
        og_smem <= 110 * 1024) {
        static std::mutex og_mu;
        static bool og_attr[64] = {false};
        CU_TRY(configure_once(og_mu, og_attr, [] {
            return cudaFuncSetAttribute(oproj_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) ==
                       cudaSuccess &&
                   cudaFuncSetAttribute(oproj_gemv_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) ==
                       cudaSuccess;
        }));
        OgParams og = {};
        og.Wo = a->Wo;
        og.obf = ap.obf;
        og.u = a->u;
        og.bl_off = a->bl_off;
        og.out = a->out;
        og.B = a->B;
        og.N = a->N;
        og.din = a->din;
        og.HD = HD;
        return launch(oproj_gemv_kernel, dim3(og_ctas), dim3(OG_THREADS), og_smem, s, og);
    }
    CUtensorMap oA[2], oW[3];
    if (!act_map(&oA[0], ap.obf, a->B, HD) || !make_map(&oW[0], a->Wo, a->din, HD, L.bn)) return WF_ERR_CUDA;
    oA[1] = oA[0];
    oW[1] = oW[2] = oW[0];
    PjParams po = proj_params(a, L, ws);
    po.num_k = cdiv(HD, BK);
    const int otiles = add_seg(po, 0, PJ_OUT, 0, 0, a->B, a->din, L.bn);
    return launch_proj(oA, oW, po, otiles, s);
}

size_t catchup_workspace_bytes(int B, int N, int din, int H, int G, int D) {
    return cu_layout(B, N, din, H, G, D).total;
}

// Shared memory an attention CTA asks for (validated on the host).
size_t catchup_attend_smem(int H, int G, int D) {
    (void)H;
    (void)G;
    const size_t stride = (size_t)D + 8;
    return 128 + AT_STAGES * (2 * (size_t)AT_PASS_ROWS * (size_t)D * 2) + 16 * stride * 2 + AT_STAGES * 8 + 16;
}

}  // namespace wf
