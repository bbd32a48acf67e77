// LM head / draft head as a tcgen05 GEMM with the selection fused into the
// epilogue: out[r] = argmax_v <act_r, W_v> (target LM head, greedy choice) or
// the top-k of the same logits (EAGLE-3 draft head).  The logits live only in
// TMEM; they are never written to memory.
//
// Per CTA (one per SM, persistent over tiles of BM activation rows x BN
// weight rows):
//   warp 0     TMA producer: stages [BK x BM] activation and [BK x BN] weight
//              boxes (128-byte swizzle) into a shared-memory ring of p.stages
//              stages (4 with several activation tiles; with one, the
//              activation slot is only as large as the box and the ring 5-6
//              stages deep, so more weight bytes are in flight per SM)
//   warp 1     allocates TMEM (2 x BN fp32 columns = two accumulators) and one
//              elected lane issues tcgen05.mma (M=128, N = the tile's weight
//              rows <= 256, K=16) per stage
//   warps 2-5  epilogue: tcgen05.ld the finished accumulator (thread = one
//              activation row, 32 columns per load), keep the running best
//              (argmax; a pairwise tree per 32 columns where the last tile's
//              scan is exposed) or a sorted top-k per row, and release the
//              accumulator so the next tile's MMAs overlap this scan.
// With one activation tile, each weight matrix is cut into a multiple of the
// CTA count of tiles of two heights (h and h - 16), so that every CTA sweeps
// the same weight rows.
// Argmax rows are combined across CTAs with a 64-bit atomicMax on a packed
// (order-preserving logit, ~id) key; the last CTA to finish converts the keys
// to ids and resets them to zero.  Top-k rows write one sorted candidate list
// per tile; wf_topk_merge combines them.
// DUAL: one launch sweeps two problems - the target LM head (argmax) and the
// EAGLE-3 draft head (top-k) - through the same pipeline, so the smaller draft
// matrix streams with the larger one instead of as a second, under-filled
// sweep; each CTA takes its draft-head tiles first, so that its last tile has
// the cheap epilogue.  One activation tile each, or (with paired CTAs) the
// LM head's tile pairs plus the draft head's rows in one tile pair.  A
// draft-head tile keeps a 10-wide candidate list when k <= 10, else 16.
//
// Every wait is bounded: a wait that runs out records WF_ERR_TIMEOUT, raises a
// CTA-wide abort flag, drains its own in-flight copies / MMAs (again bounded)
// and the CTA frees TMEM and exits.
#include <cudaTypedefs.h>

#include "wf_internal.cuh"
#include "wf_merge.cuh"

namespace wf {

constexpr int STAGES = 4;             // ring depth with several activation tiles
constexpr int STAGES_MAX = 8;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int GEMM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;     // two fp32 accumulators of BN columns
// Ring bytes with one activation tile: leaves room on the SM for the small
// CTAs that run beside the sweep (the router over every row of a short round).
constexpr int RING_BUDGET = 210 * 1024;
// Activation bytes a paired sweep keeps in L2 while the weights stream past.
constexpr long PAIR_GROUP_BYTES = 48L << 20;
// Paired-CTA sweeps run alone on their SMs: seven stages of 32 KB.
constexpr int RING_BUDGET_PAIR = 224 * 1024;
constexpr int GEMM_SMEM_MAX = RING_BUDGET_PAIR + 1024 + 256;
constexpr int KT_TOPK = WF_MAX_TOPK;
// A narrower candidate list for k <= 10 (EAGLE-3's top-10): a tile's list is
// its 10 best, so an insertion shifts 9 entries instead of 15 and fewer
// logits clear the list's smallest entry.
constexpr int KT_TOPK10 = 10;
MergeArgs merge_args(int B, int Vd, int num_n, int k, const int32_t* d2t, int32_t* draft_ids, int32_t* tids,
                     float* vals, void* ws, size_t cand_off, float* lse = nullptr, size_t lsep_off = 0);
wf_status launch_topk_merge(const MergeArgs& a, void* ws, cudaStream_t s);

struct GemmParams {
    int M_rows;        // activation rows (P or B)
    int N_w;           // weight rows (V or Vd)
    int num_m, num_n, num_k;
    int stages;        // ring stages (<= STAGES_MAX)
    int stage_bytes;   // activation slot + weight slot (a multiple of 1024)
    int a_alloc;       // activation slot bytes (a multiple of 1024)
    int k;             // top-k count (top-k mode)
    int bn;            // weight rows per tile (UMMA N): a multiple of 16, 128..256
    int nbig;          // tiles of bn rows; the other num_n - nbig tiles have bn - 16 (big ones first)
    uint32_t idesc;    // instruction descriptor for M = BM, N = bn
    uint32_t idesc_s;  // ... N = bn - 16
    int weight_evict_first;
    int group;         // activation tiles (pairs of them with PAIR) swept against every weight tile before the next group
    int a_bytes;       // bytes one activation box delivers (box rows x 128 B)
    uint64_t* keys;    // argmax: [M_rows] packed keys, zero on entry, zero on exit
    int32_t* ids;      // argmax: [M_rows] out
    float* maxlogit;   // argmax: [M_rows] out or null
    uint64_t* cand;    // top-k: [tiles][BM][k]
    float2* lsep;      // top-k: [tiles][BM] (max, sum e^(logit - max)) over the tile's columns, or null
    float4* ent;       // entropy: [M_rows][CTA slots] running (max, sum e^z, sum z e^z), z = logit - max
    float* H;          // entropy: [M_rows] out
    int ent_defer;     // entropy: leave the statistics for the acceptance step to merge at the accepted rows
    int32_t* route;    // entropy: [M_rows] out (H > tau) or null
    float tau;
    const int32_t* src_rows;   // entropy over gathered rows: the source row of each, or null
    int src_P;
    // DUAL: the second problem (top-k, one activation tile) whose num_n2 tiles
    // follow the first problem's; its candidate lists go to cand
    int M_rows2, N_w2, num_n2, a_bytes2;
    int bn2, nbig2;             // its tile heights: nbig2 of bn2 rows, the rest bn2 - 16 (big ones last)
    uint32_t idesc2, idesc2_s;
    Control* ctrl;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void gemm_fail(Control* ctrl, volatile int* abort_flag, uint32_t where) {
    *abort_flag = 1;
    record_error(ctrl, WF_ERR_TIMEOUT, where);
}


// Insert (v, id) into a descending list of KT entries (earlier entry wins ties).
template <int KT>
__device__ __forceinline__ void topk_insert(float (&tv)[KT], int (&ti)[KT], float v, int id) {
#pragma unroll
    for (int j = KT - 1; j > 0; --j) {
        const bool shift = tv[j - 1] < v;
        const bool land = !shift && tv[j] < v;
        tv[j] = shift ? tv[j - 1] : (land ? v : tv[j]);
        ti[j] = shift ? ti[j - 1] : (land ? id : ti[j]);
    }
    if (tv[0] < v) {
        tv[0] = v;
        ti[0] = id;
    }
}

// Weight rows of tile n of a problem with num_n tiles: nbig of them are bn
// rows high, the others bn - 16 (all bn when nbig = num_n), the big ones first
// or last.  Two heights let the tile count be a multiple of the CTA count, so
// that every CTA sweeps the same number of weight rows within 16 a tile.
struct TileSpan {
    int row0, rows;
    bool big;
};
__device__ __forceinline__ TileSpan tile_span(int n, int num_n, int bn, int nbig, bool big_first) {
    const int ns = num_n - nbig;
    if (big_first) {
        if (n < nbig) return {n * bn, bn, true};
        return {nbig * bn + (n - nbig) * (bn - 16), bn - 16, false};
    }
    if (n < ns) return {n * (bn - 16), bn - 16, false};
    return {ns * (bn - 16) + (n - ns) * bn, bn, true};
}

// Fold the columns j < lim of one 32-column chunk into a row's running
// softmax statistics; tv0 is the row's largest column so far in this tile,
// this chunk included, and em the largest before the tile, so a new running
// maximum shows in tv0.  Sums run in base 2: z = (v - em) log2 e, es = sum
// 2^z (the same terms as sum e^(v - em)), et = sum z 2^z (ln 2 times the
// natural-log sum; scaled back when published).
__device__ __forceinline__ void ent_fold(const uint32_t (&r)[32], int lim, float tv0, float& em, float& es,
                                         float& et) {
    if (tv0 > em) {   // new running maximum: rescale what was summed so far
        if (es > 0.f) {
            const float dz = (em - tv0) * LOG2E;
            const float sc = ex2_approx(dz);
            et = (et + dz * es) * sc;
            es *= sc;
        }
        em = tv0;
    }
    const float off = em * LOG2E;
    // four interleaved partial sums: the adds of one chunk form four short
    // chains instead of one 32 long
    float s4[4] = {0.f, 0.f, 0.f, 0.f}, t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j < lim) {
            const float z = fmaf(__uint_as_float(r[j]), LOG2E, -off);
            const float e = ex2_approx(z);
            s4[j & 3] += e;
            t4[j & 3] = fmaf(z, e, t4[j & 3]);
        }
    es += (s4[0] + s4[1]) + (s4[2] + s4[3]);
    et += (t4[0] + t4[1]) + (t4[2] + t4[3]);
}

// Fold the columns j < lim of one chunk into a row's running (max lm, sum
// ls = sum e^(v - lm)) over one tile; tv0 is the tile's largest column so far,
// this chunk included.  Sums run in base 2 (the same terms: 2^((v - lm) log2 e)).
__device__ __forceinline__ void lse_fold(const uint32_t (&r)[32], int lim, float tv0, float& lm, float& ls) {
    if (tv0 > lm) {
        if (ls > 0.f) ls *= ex2_approx((lm - tv0) * LOG2E);
        lm = tv0;
    }
    const float off = lm * LOG2E;
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j < lim) ls += ex2_approx(fmaf(__uint_as_float(r[j]), LOG2E, -off));
}

// One finished accumulator as epilogue thread rit sees it (activation row
// m * BM + rit of a problem with M_rows rows and N_w weight rows): wait for
// it, keep the row's best (KT = 1) or top KT over the tile's columns and, with
// ENT, fold the columns into the row's softmax statistics; hand the
// accumulator back to the MMA warp, then publish the row's result (a packed
// key for argmax, the tile's sorted candidate list for top-k).
// tempty_first: in the second CTA of a pair, the shared::cluster address of
// the first CTA's accumulator-empty barriers (the first CTA issues the MMAs
// into both CTAs' TMEM); 0 otherwise.
template <int KT, bool ENT, bool TAIL>
__device__ __forceinline__ bool epilogue_tile(const GemmParams& p, uint64_t* tfull, uint64_t* tempty,
                                              uint32_t tempty_first, volatile int* abort_flag, uint32_t tmem_base,
                                              uint32_t tile_i, int q, int rit, int M_rows, int N_w, int m, int n,
                                              const TileSpan sp, int cand_num_m, float& em, float& es, float& et) {
    static_assert(!ENT || KT == 1, "the softmax statistics ride on the argmax epilogue");
    const uint32_t acc = tile_i & 1;
    const uint32_t acc_ph = (tile_i >> 1) & 1;
    const bool quad_live = m * BM + q * 32 < M_rows;
    const int row = m * BM + rit;
    if (!mbar_wait(&tfull[acc], acc_ph, p.timeout_ns, abort_flag)) {
        gemm_fail(p.ctrl, abort_flag, 0x300);
        return false;
    }
    tc_fence_after();
    float tv[KT];
    int ti[KT];
#pragma unroll
    for (int j = 0; j < KT; ++j) {
        tv[j] = -INFINITY;
        ti[j] = 0;
    }
    float lm = -INFINITY, ls = 0.f;   // top-k with log-sum-exp: this tile's (max, sum e^(v - max)) of the row
    if (quad_live) {
        const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
        if constexpr (KT == 1 && TAIL) {
            // two 32-column loads in flight per wait; each chunk's best by a
            // pairwise tree over adjacent columns (a strict > keeps the lower
            // column on ties, as a left-to-right scan would)
            for (int c00 = 0; c00 < sp.rows; c00 += 64) {
                uint32_t r2[2][32];
                const bool two = c00 + 32 < sp.rows;   // the same for the whole warp
                tmem_ld_32x32b_x32(tbase + c00, r2[0]);
                if (two) tmem_ld_32x32b_x32(tbase + c00 + 32, r2[1]);
                tmem_ld_wait();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (hh == 1 && !two) break;
                    const uint32_t (&r)[32] = r2[hh];
                    const int c0 = c00 + 32 * hh;
                    const int col0 = sp.row0 + c0;
                    // columns >= lim are past the weight matrix or past this tile; rows
                    // past the activations (stale shared-memory rows) take no part
                    const int lim = row < M_rows ? min(N_w - col0, sp.rows - c0) : 0;
                    float bv[16];
                    int bj[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float a = 2 * j < lim ? __uint_as_float(r[2 * j]) : -INFINITY;
                        const float b = 2 * j + 1 < lim ? __uint_as_float(r[2 * j + 1]) : -INFINITY;
                        const bool t = b > a;
                        bv[j] = t ? b : a;
                        bj[j] = t ? 2 * j + 1 : 2 * j;
                    }
#pragma unroll
                    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                        for (int j = 0; j < w; ++j) {
                            const bool t = bv[2 * j + 1] > bv[2 * j];
                            bv[j] = t ? bv[2 * j + 1] : bv[2 * j];
                            bj[j] = t ? bj[2 * j + 1] : bj[2 * j];
                        }
                    if (bv[0] > tv[0]) {
                        tv[0] = bv[0];
                        ti[0] = col0 + bj[0];
                    }
                    if constexpr (ENT) ent_fold(r, lim, tv[0], em, es, et);
                }
            }
        } else {
            // one load per wait and a left-to-right scan: fewer registers and
            // TMEM reads beside the MMAs of a tensor-bound sweep, whose tiles
            // are long enough to hide the epilogue
            const bool want_lse = KT > 1 && p.lsep != nullptr;
            for (int c0 = 0; c0 < sp.rows; c0 += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + c0, r);
                tmem_ld_wait();
                const int col0 = sp.row0 + c0;
                const int lim = row < M_rows ? min(N_w - col0, sp.rows - c0) : 0;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float v = __uint_as_float(r[j]);
                    if (j < lim) {
                        if constexpr (KT == 1) {
                            if (v > tv[0]) {
                                tv[0] = v;
                                ti[0] = col0 + j;
                            }
                        } else {
                            if (v > tv[KT - 1]) topk_insert<KT>(tv, ti, v, col0 + j);
                        }
                    }
                }
                if constexpr (ENT) ent_fold(r, lim, tv[0], em, es, et);
                if (want_lse) lse_fold(r, lim, tv[0], lm, ls);
            }
        }
    }
    tc_fence_before();
    if (tempty_first)
        mbar_arrive_remote(tempty_first + acc * (uint32_t)sizeof(uint64_t), 1u);
    else
        mbar_arrive(&tempty[acc]);
    if (quad_live && row < M_rows) {
        if constexpr (KT == 1) {
            atomicMax(reinterpret_cast<unsigned long long*>(p.keys + row),
                      (unsigned long long)pack_key(tv[0], (uint32_t)ti[0]));
        } else {
            const size_t t = (size_t)n * cand_num_m + m;   // the candidate list of tile (m, n)
            uint64_t* dst = p.cand + (t * BM + rit) * p.k;
            for (int j = 0; j < KT; ++j)
                if (j < p.k) dst[j] = tv[j] == -INFINITY ? 0ull : pack_key(tv[j], (uint32_t)ti[j]);
            if (p.lsep) p.lsep[t * BM + rit] = make_float2(lm, ls);
        }
    }
    return true;
}

// Tile u of the first problem -> (activation tile, or pair of them, mt; weight
// tile n).  The activation tiles are taken in groups of `group`: every weight
// tile meets one group's tiles before the next group starts, so a group's
// activations stay in L2 while the weights stream past (the weights are read
// once per group).  group >= num_mt gives the plain order u = n * num_mt + mt.
struct TileMN {
    int mt, n;
};
__device__ __forceinline__ TileMN tile_mn(int u, int num_mt, int num_n, int group) {
    const int per = group * num_n;
    const int g = u / per;
    const int first = g * group;
    const int size = min(group, num_mt - first);
    const int r = u - g * per;
    return {first + r % size, r / size};
}

// Tile u of the v-th position in the schedule.  DUAL: the second problem's
// tiles (u >= U0, top-k, the costlier epilogue) come first, so that a CTA's
// last tile, whose epilogue nothing overlaps, is an argmax tile.  Each tile
// stays with the same CTA as in plain order when both problems' tile counts
// are multiples of the CTA count (balanced tiles); otherwise the CTAs still
// split the tiles exactly once between them.
template <bool DUAL>
__device__ __forceinline__ int tile_order(int v, int U0, int U) {
    if constexpr (!DUAL) return v;
    const int n2 = U - U0;
    return v < n2 ? U0 + v : v - n2;
}

// Each CTA loads its own activation and weight boxes; tiles (m, n) are visited
// in the order t = n * num_m + m, so the CTAs working at the same time share
// the weight tile through L2.
// PAIR (several activation tiles, no ENT): clusters of two CTAs take
// tile pairs (m, n), (m + 1, n) with one paired MMA of M = 256 rows: each CTA
// loads its own activation tile and half of the weight tile (its bytes are
// counted on the first CTA's stage barrier), the first CTA issues every MMA
// and commits to both CTAs' barriers, and each CTA's epilogue reads its own
// TMEM rows.  A weight byte crosses the L2 -> SM crossbar and is read from
// shared memory once per pair.
// ENT (with KT = 1): also accumulate, per row, the softmax statistics of the
// logits so that the entropy of the next-token distribution comes out of the
// same weight sweep.  Needs every CTA's rows fixed over its tiles: at most two
// activation tiles, and a grid that is a multiple of their count or, with
// PAIR, exactly two of them (each CTA of a pair keeps its own).
// DUAL (with KT = 1): tiles U0.. are the second problem's
// (activation map tmA2, weight map tmB2, top-k into p.cand), swept first
// (tile_order); with ENT the first problem's tiles also feed the entropy
// statistics; with PAIR they are pair tiles over the second problem's rows
// (at most 2 BM: each CTA its own half).
// The plain argmax sweep (<1, false, false, false>) runs beside the router
// kernel at batch 1 and must stay within 96 registers a thread: two of its
// warps and two 160-register router warps then fill one SM sub-partition's
// 16K registers exactly (at 104 the router waits for the sweep to finish).
template <int KT, bool ENT, bool DUAL, bool PAIR>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_select_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                       const __grid_constant__ CUtensorMap tmBs, const __grid_constant__ CUtensorMap tmB2s,
                       const GemmParams p) {
    static_assert(!DUAL || KT == 1, "the dual sweep pairs an argmax head with a top-k head");
    extern __shared__ uint8_t smem_raw[];
    // ENT needs every CTA's rows fixed over its tiles: with PAIR that holds
    // for two activation tiles (each CTA of a pair keeps tile `rank`) only
    if (ENT && PAIR && p.num_m > 2) {   // the host never launches this; both CTAs of a pair leave
        if (threadIdx.x == 0) record_error(p.ctrl, WF_ERR_UNSUPPORTED, 0x330);
        return;
    }
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stages = p.stages;
    // stage s: activation slot at s * stage_bytes, weight slot a_alloc bytes on
    // (the MMA reads BM activation rows; past a short box those are the same
    // stage's weight rows, which only feed accumulator rows nobody keeps)
    auto stA = [&](int st) { return smem + (size_t)st * p.stage_bytes; };
    auto stB = [&](int st) { return smem + (size_t)st * p.stage_bytes + p.a_alloc; };
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * p.stage_bytes);
    uint64_t* empty = full + STAGES_MAX;
    uint64_t* tfull = empty + STAGES_MAX;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* last_flag = reinterpret_cast<int*>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // tiles: u -> (activation tile m = u % num_m, weight tile n = u / num_m);
    // PAIR: u -> activation tiles 2 (u % num_mt) + rank of the pair, weight tile u / num_mt
    const int rank = PAIR ? (int)(cluster_ctarank() & 1u) : 0;
    const bool first = rank == 0;   // PAIR: the CTA that issues the MMAs
    const int slot = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int nslots = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int num_m = p.num_m;
    const int num_mt = PAIR ? (num_m + 1) >> 1 : num_m;
    const int U0 = num_mt * p.num_n;
    const int U = U0 + (DUAL ? p.num_n2 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], PAIR ? 256 : 128);   // PAIR: both CTAs' epilogue threads release
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (p.nbig < p.num_n) tma_prefetch_desc(&tmBs);
        if constexpr (DUAL) {
            tma_prefetch_desc(&tmA2);
            tma_prefetch_desc(&tmB2);
            if (p.nbig2 < p.num_n2) tma_prefetch_desc(&tmB2s);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // both CTAs' barriers and TMEM exist before either uses the other's
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above overlaps the previous kernel on the stream; inputs and
    // the workspace are touched only after it has finished.  Then the next
    // kernel may be scheduled (everything before this one is complete by now).
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = p.weight_evict_first ? policy_evict_first() : policy_evict_normal();
            const uint64_t pol_a = policy_evict_last();
            // PAIR: both CTAs' copies of a stage are counted on the first CTA's barrier
            const uint32_t full_first = PAIR ? cluster_addr(&full[0], 0) : 0;
            uint32_t it = 0;  // stages issued so far
            int s = 0;        // = it % stages
            uint32_t ph = 0;  // = (it / stages) & 1
            bool ok = true;
            for (int v = slot; v < U && ok; v += nslots) {
                const int u = tile_order<DUAL>(v, U0, U);
                const bool second = DUAL && u >= U0;
                const TileMN tm = tile_mn(second ? 0 : u, num_mt, p.num_n, p.group);
                const int m = second ? (PAIR ? rank : 0) : (PAIR ? 2 * tm.mt + rank : tm.mt);
                const int n = second ? u - U0 : tm.n;
                const TileSpan sp = second ? tile_span(n, p.num_n2, p.bn2, p.nbig2, false)
                                           : tile_span(n, p.num_n, p.bn, p.nbig, true);
                const CUtensorMap* mA = second ? &tmA2 : &tmA;
                const CUtensorMap* mB = second ? (sp.big ? &tmB2 : &tmB2s) : (sp.big ? &tmB : &tmBs);
                const int wrows = PAIR ? sp.rows / 2 : sp.rows;   // weight rows this CTA loads
                const uint32_t tx = PAIR ? 2u * (uint32_t)((second ? p.a_bytes2 : p.a_bytes) + wrows * BK * 2)
                                         : (uint32_t)((second ? p.a_bytes2 : p.a_bytes) + sp.rows * BK * 2);
                for (int kc = 0; kc < p.num_k; ++kc, ++it) {
                    if (it > 0) {
                        if (++s == stages) {
                            s = 0;
                            ph ^= 1;
                        }
                    }
                    if (!mbar_wait(&empty[s], ph ^ 1, p.timeout_ns, abort_flag)) {
                        gemm_fail(p.ctrl, abort_flag, 0x100 + s);
                        ok = false;
                        break;
                    }
                    if constexpr (PAIR) {
                        if (first) mbar_arrive_expect_tx(&full[s], tx);
                        const uint32_t bar = full_first + (uint32_t)(s * sizeof(uint64_t));
                        tma_load_2d_pair(stA(s), mA, bar, kc * BK, m * BM, pol_a);
                        tma_load_2d_pair(stB(s), mB, bar, kc * BK, sp.row0 + rank * wrows, pol_w);
                    } else {
                        mbar_arrive_expect_tx(&full[s], tx);
                        tma_load_2d(stA(s), mA, &full[s], kc * BK, m * BM, pol_a);
                        tma_load_2d(stB(s), mB, &full[s], kc * BK, sp.row0, pol_w);
                    }
                }
            }
            if (!ok || *abort_flag) {
                // let every copy this thread issued land before the CTA exits
                if (!PAIR || first) {
                    for (uint32_t j = (it > (uint32_t)stages ? it - stages : 0); j < it; ++j)
                        mbar_wait(&full[j % stages], (j / stages) & 1, p.timeout_ns, nullptr);
                } else {
                    // the second CTA's copies are counted on the first CTA's
                    // barriers, which it cannot wait on: give them a fixed
                    // 200 us (a copy from L2 or HBM takes a few)
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 200000ull) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && first) {
            // PAIR: the first CTA's commits arrive on both CTAs' barriers
            const uint32_t empty_peer = PAIR ? cluster_addr(&empty[0], 1) : 0;
            const uint32_t tfull_peer = PAIR ? cluster_addr(&tfull[0], 1) : 0;
            uint32_t it = 0, tile_i = 0;
            int s = 0;        // = it % stages
            uint32_t ph = 0;  // = (it / stages) & 1
            bool ok = true, issued = false;
            for (int v = slot; v < U && ok; v += nslots, ++tile_i) {
                const int u = tile_order<DUAL>(v, U0, U);
                const bool second = DUAL && u >= U0;
                const int n = second ? u - U0 : tile_mn(u, num_mt, p.num_n, p.group).n;
                const TileSpan sp = second ? tile_span(n, p.num_n2, p.bn2, p.nbig2, false)
                                           : tile_span(n, p.num_n, p.bn, p.nbig, true);
                const uint32_t idesc = second ? (sp.big ? p.idesc2 : p.idesc2_s) : (sp.big ? p.idesc : p.idesc_s);
                const uint32_t acc = tile_i & 1;
                const uint32_t acc_ph = (tile_i >> 1) & 1;
                // PAIR: released by both CTAs' epilogues (the second's arrivals are remote)
                if (!(PAIR ? mbar_wait_cluster(&tempty[acc], acc_ph ^ 1, p.timeout_ns, abort_flag)
                           : mbar_wait(&tempty[acc], acc_ph ^ 1, p.timeout_ns, abort_flag))) {
                    gemm_fail(p.ctrl, abort_flag, 0x200);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kc = 0; kc < p.num_k; ++kc, ++it) {
                    if (it > 0) {
                        if (++s == stages) {
                            s = 0;
                            ph ^= 1;
                        }
                    }
                    if (!mbar_wait(&full[s], ph, p.timeout_ns, abort_flag)) {
                        gemm_fail(p.ctrl, abort_flag, 0x210 + s);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = umma_desc_sw128(smem_u32(stA(s)));
                    const uint64_t bdesc = umma_desc_sw128(smem_u32(stB(s)));
                    if constexpr (PAIR) {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kc | kk) != 0);
                        umma_commit_pair(smem_u32(&empty[s]));
                        umma_commit_pair(empty_peer + (uint32_t)(s * sizeof(uint64_t)));
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes of K per step (encoded >> 4)
                            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kc | kk) != 0);
                        umma_commit(&empty[s]);
                    }
                    issued = true;
                }
                if (ok) {
                    if constexpr (PAIR) {
                        umma_commit_pair(smem_u32(&tfull[acc]));
                        umma_commit_pair(tfull_peer + acc * (uint32_t)sizeof(uint64_t));
                    } else {
                        umma_commit(&tfull[acc]);
                    }
                }
            }
            if (issued && (!ok || PAIR)) {
                // every MMA issued above (PAIR: into both CTAs' TMEM) has
                // completed before TMEM is freed
                if constexpr (PAIR)
                    umma_commit_pair(smem_u32(drain));
                else
                    umma_commit(drain);
                mbar_wait(drain, 0, p.timeout_ns, nullptr);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int rit = q * 32 + lane;
        float em = -INFINITY, es = 0.f, et = 0.f;   // ENT: this row's running softmax statistics
        const uint32_t tempty_first = (PAIR && !first) ? cluster_addr(&tempty[0], 0) : 0;
        uint32_t tile_i = 0;
        for (int v = slot; v < U; v += nslots, ++tile_i) {
            const int u = tile_order<DUAL>(v, U0, U);
            bool ok;
            if (DUAL && u >= U0) {
                // the second problem's tile: top-k candidates (a 10-wide list when k <= 10);
                // PAIR: this CTA's half of the rows, lists per activation tile of the second problem
                const TileSpan sp2 = tile_span(u - U0, p.num_n2, p.bn2, p.nbig2, false);
                const int m2 = PAIR ? rank : 0, nm2 = PAIR ? (p.M_rows2 + BM - 1) / BM : 1;
                ok = p.k <= KT_TOPK10
                         ? epilogue_tile<KT_TOPK10, false, false>(p, tfull, tempty, tempty_first, abort_flag,
                                                                  tmem_base, tile_i, q, rit, p.M_rows2, p.N_w2, m2,
                                                                  u - U0, sp2, nm2, em, es, et)
                         : epilogue_tile<KT_TOPK, false, false>(p, tfull, tempty, tempty_first, abort_flag, tmem_base,
                                                                tile_i, q, rit, p.M_rows2, p.N_w2, m2, u - U0, sp2,
                                                                nm2, em, es, et);
            } else if (!PAIR && num_m == 1)   // the weight-streaming sweep: the last tile's scan is exposed
                ok = epilogue_tile<KT, ENT, true>(p, tfull, tempty, 0, abort_flag, tmem_base, tile_i, q, rit,
                                                  p.M_rows, p.N_w, 0, u, tile_span(u, p.num_n, p.bn, p.nbig, true), 1,
                                                  em, es, et);
            else {
                const TileMN tm = tile_mn(u, num_mt, p.num_n, p.group);
                ok = epilogue_tile<KT, ENT, false>(p, tfull, tempty, tempty_first, abort_flag, tmem_base, tile_i, q,
                                                   rit, p.M_rows, p.N_w, PAIR ? 2 * tm.mt + rank : tm.mt, tm.n,
                                                   tile_span(tm.n, p.num_n, p.bn, p.nbig, true), num_m, em, es, et);
            }
            if (!ok) break;
        }
        if constexpr (ENT) {
            // this CTA's rows are fixed (the grid is a multiple of num_m); publish
            // their statistics, and an empty state (S = 0) for the other
            // activation tile's rows, so that every slot a merge reads was
            // written by this launch
            for (int mm = 0; mm < num_m; ++mm) {
                const int row = mm * BM + rit;
                if (PAIR && mm != rank) continue;   // the pair's other CTA writes those rows' slot
                if (row < p.M_rows)
                    p.ent[(size_t)row * nslots + slot] =
                        PAIR || mm == slot % num_m ? make_float4(em, es, et * LN2, 0.f)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (KT == 1 && !*abort_flag) {
            // last CTA to finish turns the keys into ids and zeroes them again
            __threadfence();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (threadIdx.x == 64) {
                const uint32_t prev = atomicAdd(&p.ctrl->gemm_done, 1u);
                *last_flag = (prev == gridDim.x - 1);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (*last_flag) {
                __threadfence();
                for (int r = threadIdx.x - 64; r < p.M_rows; r += 128) {
                    const uint64_t key = __ldcg(reinterpret_cast<const unsigned long long*>(p.keys + r));
                    if (p.ids) p.ids[r] = key ? (int32_t)key_id(key) : -1;
                    if (p.maxlogit) p.maxlogit[r] = key ? key_val(key) : __int_as_float(0x7fc00000);
                    p.keys[r] = 0;
                }
                if (threadIdx.x == 64) p.ctrl->gemm_done = 0;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (ENT && KT == 1) {
        // The last CTA: entropy per row from every CTA's softmax statistics,
        // merged in a fixed order (each lane its slots in increasing order, then
        // a fixed shuffle tree), H = log S - T / S.  All of its warps take part,
        // ENT_RB rows each at a time: every slot load in flight before any is
        // used (a row's slots are contiguous, so each load is coalesced), the
        // rows' merge chains interleaved, and lane q finishing row q.
        if (*last_flag && !p.ent_defer) {
            static_assert(ENT_MAX_SLOTS % 32 == 0, "slots are shared out evenly over the lanes");
            constexpr int SPL = ENT_MAX_SLOTS / 32;   // slots per lane
            constexpr int ENT_RB = 4;
            constexpr int NW = GEMM_THREADS / 32;
            __threadfence();   // after the epilogue warps' arrival count: read every CTA's slots
            for (int r0 = warp * ENT_RB; r0 < p.M_rows; r0 += NW * ENT_RB) {
                const int rl = r0 + lane;   // the row lane q < ENT_RB finishes
                // gathered rows: a source row outside [0, src_P) has no entropy
                const int src = (p.src_rows && lane < ENT_RB && rl < p.M_rows) ? p.src_rows[rl] : 0;
                float4 st[ENT_RB][SPL];
#pragma unroll
                for (int q = 0; q < ENT_RB; ++q)
#pragma unroll
                    for (int i = 0; i < SPL; ++i) {
                        const int r = r0 + q, sl = lane + 32 * i;
                        st[q][i] = (r < p.M_rows && sl < nslots) ? __ldcg(p.ent + (size_t)r * nslots + sl)
                                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                float M[ENT_RB], S[ENT_RB], T[ENT_RB];
#pragma unroll
                for (int q = 0; q < ENT_RB; ++q) {
                    M[q] = -INFINITY;
                    S[q] = 0.f;
                    T[q] = 0.f;
#pragma unroll
                    for (int i = 0; i < SPL; ++i) ent_merge(M[q], S[q], T[q], st[q][i].x, st[q][i].y, st[q][i].z);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                    for (int q = 0; q < ENT_RB; ++q) {
                        const float m2 = __shfl_xor_sync(0xffffffffu, M[q], off);
                        const float s2 = __shfl_xor_sync(0xffffffffu, S[q], off);
                        const float t2 = __shfl_xor_sync(0xffffffffu, T[q], off);
                        ent_merge(M[q], S[q], T[q], m2, s2, t2);
                    }
                // every lane holds every row's totals; lane q takes row r0 + q
                float Sq = S[0], Tq = T[0];
#pragma unroll
                for (int q = 1; q < ENT_RB; ++q)
                    if (lane == q) {
                        Sq = S[q];
                        Tq = T[q];
                    }
                if (lane < ENT_RB && rl < p.M_rows) {
                    const bool bad = p.src_rows && (src < 0 || src >= p.src_P);
                    const float h = bad ? __int_as_float(0x7fc00000) : logf(Sq) - Tq / Sq;
                    p.H[rl] = h;
                    if (p.route) p.route[rl] = bad ? -1 : (h > p.tau ? 1 : 0);
                }
                // leave the workspace zeroed (after the loads are used: a store
                // to an address with a load still in flight waits for it)
#pragma unroll
                for (int q = 0; q < ENT_RB; ++q)
#pragma unroll
                    for (int i = 0; i < SPL; ++i) {
                        const int r = r0 + q, sl = lane + 32 * i;
                        if (r < p.M_rows && sl < nslots)
                            p.ent[(size_t)r * nslots + sl] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
            }
        }
    }
    if constexpr (PAIR) cluster_sync();   // the first CTA's MMAs and the second's remote arrivals are done
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// --------------------------------------------------------------------- top-k merge
// One CTA per activation row (wf_merge.cuh).
__global__ void __launch_bounds__(MERGE_THREADS) topk_merge_kernel(const MergeArgs a, Control* ctrl) {
    __shared__ uint64_t wbest[MERGE_SCRATCH];
    pdl_wait();
    pdl_trigger();
    topk_merge_row<12>(a, blockIdx.x, wbest, ctrl);
}

// --------------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// [rows, cols] bf16 row-major; boxes of 64 columns (128 B, swizzled) x box_rows rows.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms();

// Weight rows per tile.  Several activation tiles: 256 (largest operand reuse).
// One activation tile (the weight-streaming case): the multiple of 16 in
// [BN_MIN, 256] that minimises the busiest CTA's rows, waves x (bn + 16) - the
// 16 standing for a tile's fixed cost - so the last wave is not left mostly
// idle.  N_w2 > 0: a second weight matrix swept in the same launch.
static int pick_bn(int num_m, int N_w, int sms, int N_w2 = 0) {
    if (num_m > 1) return BN;
    int best = BN;
    long best_cost = -1;
    for (int bn = BN; bn >= BN_MIN; bn -= 16) {
        const long tiles = cdiv(N_w, bn) + (N_w2 > 0 ? cdiv(N_w2, bn) : 0);
        const long waves = cdiv(tiles, sms);
        const long cost = waves * (bn + 16);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

// Balanced tiles for one weight matrix swept by `sms` CTAs with one
// activation tile: the fewest tiles of at most BN rows whose count is a
// multiple of sms, nbig of them bn rows high and the rest bn - 16, so that the
// round-robin tile schedule gives every CTA the same number of tiles and the
// same weight rows within 16 a tile.  False when a CTA would get fewer than
// BN_MIN rows (pick_bn's uniform tiles are used then).
struct TileGeom {
    int num_n, bn, nbig;
};
static bool balanced_tiles(int N_w, int sms, TileGeom* g) {
    if (sms < 1 || N_w < sms * BN_MIN) return false;
    const int T = sms * cdiv(N_w, sms * BN);
    const int hs = N_w / T / 16 * 16;   // the average height, rounded down to 16
    g->num_n = T;
    if (T * hs == N_w) {
        g->bn = hs;
        g->nbig = T;
    } else {
        g->bn = hs + 16;
        g->nbig = cdiv(N_w - T * hs, 16);   // the last tile may reach up to 15 rows past the matrix
    }
    return true;
}

// The shared-memory ring: with several activation tiles, STAGES stages of a
// full activation box and a full weight box; with one, an activation slot as
// large as its box (a_rows x 128 bytes) and as many stages as RING_BUDGET
// holds.  Returns the dynamic shared memory of the launch.
// Paired-CTA sweeps: the weight slot holds half a tile (BN / 2 rows), so the
// same budget holds six stages.
static int set_ring(GemmParams& p, int one_tile_a_rows, bool pair = false) {
    const int b_bytes = pair ? B_BYTES / 2 : B_BYTES;
    if (one_tile_a_rows <= 0 && !pair) {
        p.a_alloc = A_BYTES;
        p.stages = STAGES;
    } else {
        p.a_alloc = one_tile_a_rows > 0 ? one_tile_a_rows * BK * 2 : A_BYTES;   // a multiple of 1024
        int st = (pair ? RING_BUDGET_PAIR : RING_BUDGET) / (p.a_alloc + b_bytes);
        p.stages = st < STAGES ? STAGES : (st > STAGES_MAX ? STAGES_MAX : st);
    }
    p.stage_bytes = p.a_alloc + b_bytes;
    return p.stages * p.stage_bytes + 1024 + 256;
}

// Clusters of two paired-CTA sweep CTAs that can be resident at once (queried
// once per device).  DUAL: the sweep that also carries the draft head.
template <int KT, bool DUAL = false, bool ENT = false>
static int pair_slots(int smem) {
    static std::mutex mu;
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return num_sms() / 2;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && cached[dev]) return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 64);
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_select_kernel<KT, ENT, DUAL, true>, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = num_sms() / 2;
    }
    if (dev < 64) cached[dev] = n;
    return n;
}

template <int KT, bool ENT>
static wf_status launch_select(const uint16_t* act, int M_rows, const uint16_t* W, int N_w, int d, GemmParams p,
                               cudaStream_t s, int* num_n_out = nullptr, int* grid_out = nullptr) {
    static std::mutex mu;
    static bool attr_set[64] = {false};
    const wf_status cst = configure_once(mu, attr_set, [] {
        return cudaFuncSetAttribute(gemm_select_kernel<KT, ENT, false, false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_MAX) == cudaSuccess &&
               cudaFuncSetAttribute(gemm_select_kernel<KT, ENT, false, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_MAX) == cudaSuccess;
    });
    if (cst != WF_OK) return cst;
    CUtensorMap ta, tb, tbs;
    const int num_m = cdiv(M_rows, BM);
    if (ENT && num_m > 2) return WF_ERR_UNSUPPORTED;
    // several activation tiles: CTA pairs with the paired MMA (M = 256), each
    // loading half of every weight tile
    const bool pair = num_m > 1 && (!ENT || num_m == 2);
    // With a single activation tile the box covers only the rows that exist
    // (rounded up to a whole 8-row swizzle atom): no zero rows cross the
    // crossbar.  The UMMA still reads all BM rows of the stage; rows past the
    // box hold stale data and produce accumulator rows the epilogue never keeps.
    const int a_rows = num_m == 1 ? (M_rows + 7) / 8 * 8 : BM;
    if (!make_map(&ta, act, (uint64_t)M_rows, (uint64_t)d, (uint32_t)a_rows)) return WF_ERR_CUDA;
    TileGeom tg;
    if (balanced_tiles(N_w, num_sms(), &tg)) {
        p.num_n = tg.num_n;
        p.bn = tg.bn;
        p.nbig = tg.nbig;
    } else {
        p.bn = pick_bn(num_m, N_w, num_sms());
        p.num_n = cdiv(N_w, p.bn);
        p.nbig = p.num_n;
    }
    const int bn = p.bn;
    const int split = pair ? 2 : 1;   // a pair's CTAs each load half of a weight tile (bn is a multiple of 16)
    if (!make_map(&tb, W, (uint64_t)N_w, (uint64_t)d, (uint32_t)(bn / split))) return WF_ERR_CUDA;
    tbs = tb;
    if (p.nbig < p.num_n && !make_map(&tbs, W, (uint64_t)N_w, (uint64_t)d, (uint32_t)((bn - 16) / split)))
        return WF_ERR_CUDA;
    if (num_n_out) *num_n_out = p.num_n;
    p.M_rows = M_rows;
    p.N_w = N_w;
    p.num_m = num_m;
    p.idesc = umma_idesc_bf16(split * BM, bn);
    p.idesc_s = p.nbig < p.num_n ? umma_idesc_bf16(split * BM, bn - 16) : p.idesc;
    p.num_k = cdiv(d, BK);
    // Weight tiles are read by every activation tile at about the same time and
    // never again: first out of L2, so that the activations (read once per
    // weight tile; 80 MB for 15,616 rows) stay resident.
    p.weight_evict_first = 1;
    // paired sweeps: activation groups of at most PAIR_GROUP_BYTES, evened out
    const int num_mt = pair ? cdiv(num_m, 2) : num_m;
    p.group = num_mt;
    if (pair) {
        const long per_mt = 2L * BM * d * 2;   // activation bytes of one tile pair
        const int most = (int)(PAIR_GROUP_BYTES / per_mt) > 0 ? (int)(PAIR_GROUP_BYTES / per_mt) : 1;
        const int groups = cdiv(num_mt, most);
        p.group = cdiv(num_mt, groups);
    }
    p.a_bytes = a_rows * BK * 2;
    p.timeout_ns = wait_timeout_ns();
    const int smem = set_ring(p, num_m == 1 ? a_rows : 0, pair);
    if (pair) {
        const int pairs = cdiv(num_m, 2) * p.num_n;
        const int slots = pair_slots<KT, false, ENT>(smem);
        const int grid = 2 * (pairs < slots ? pairs : slots);
        if (ENT && grid_out) *grid_out = grid / 2;   // ENT: the statistics' slots are the pairs
        return launch_cluster(gemm_select_kernel<KT, ENT, false, true>, dim3(grid), dim3(GEMM_THREADS), smem, s,
                              2u, ta, tb, ta, tb, tbs, tbs, p);
    }
    const int tiles = p.num_m * p.num_n;
    int grid = tiles < num_sms() ? tiles : num_sms();
    if (ENT) {   // every CTA keeps the rows of one activation tile: a grid that is a multiple of num_m
        if (grid > ENT_MAX_SLOTS) grid = ENT_MAX_SLOTS;
        grid -= grid % num_m;
    }
    if (grid_out) *grid_out = grid;
    return launch(gemm_select_kernel<KT, ENT, false, false>, dim3(grid), dim3(GEMM_THREADS), smem, s, ta, tb, ta, tb,
                  tbs, tbs, p);
}

static GemmParams params_for(void* ws) {
    GemmParams p = {};
    p.ctrl = reinterpret_cast<Control*>(ws);
    p.keys = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ws) + sizeof(Control));
    return p;
}

wf_status launch_lmhead_argmax(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                               float* maxlogit, void* ws, cudaStream_t s) {
    GemmParams p = params_for(ws);
    p.k = 1;
    p.ids = ids;
    p.maxlogit = maxlogit;
    return launch_select<1, false>(hidden, P, W, V, d, p, s);
}

// The same sweep plus the entropy of softmax(logits) per row (rows <= 2 tiles).
wf_status launch_lmhead_entropy(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                                float* maxlogit, float* H, int32_t* route, float tau, const int32_t* src_rows,
                                int src_P, void* ws, size_t ent_off, cudaStream_t s, int* defer_slots) {
    GemmParams p = params_for(ws);
    p.ent_defer = defer_slots != nullptr;
    p.k = 1;
    p.ids = ids;
    p.maxlogit = maxlogit;
    p.ent = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(ws) + ent_off);
    p.H = H;
    p.route = route;
    p.tau = tau;
    p.src_rows = src_rows;
    p.src_P = src_P;
    return launch_select<1, true>(hidden, P, W, V, d, p, s, nullptr, defer_slots);
}

wf_status launch_draft_topk(const uint16_t* x, const uint16_t* Wd, const int32_t* d2t, int B, int d, int Vd, int k,
                            int32_t* draft_ids, int32_t* tids, float* vals, float* lse, void* ws, size_t cand_off,
                            size_t lsep_off, cudaStream_t s) {
    GemmParams p = params_for(ws);
    p.k = k;
    p.cand = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ws) + cand_off);
    p.lsep = lse ? reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(ws) + lsep_off) : nullptr;
    int num_n = 0;
    wf_status st = k <= KT_TOPK10 ? launch_select<KT_TOPK10, false>(x, B, Wd, Vd, d, p, s, &num_n)
                                  : launch_select<KT_TOPK, false>(x, B, Wd, Vd, d, p, s, &num_n);
    if (st != WF_OK) return st;
    return launch_topk_merge(merge_args(B, Vd, num_n, k, d2t, draft_ids, tids, vals, ws, cand_off, lse, lsep_off),
                             ws, s);
}

// The shared sweep for rounds of several activation tiles (P > BM, B <= 2 BM):
// the paired-CTA LM head (argmax over every verified row) with the draft
// head's tiles as extra work units of the same persistent loop, swept first
// (each CTA's draft tiles: top-k candidate lists of its half of the draft
// rows; their epilogue overlaps the LM head's first main loops), instead of
// the draft head's own sweep after the round, which fills the SMs in under
// two waves.
static wf_status launch_lmhead_draft_pair(const uint16_t* hidden, const uint16_t* W, int P, int d, int V,
                                          int32_t* ids, float* maxlogit, const uint16_t* x, const uint16_t* Wd, int B,
                                          int Vd, int k, void* ws, size_t cand_off, size_t lsep_off,
                                          int* num_n2_out, cudaStream_t s) {
    static std::mutex mu;
    static bool attr_set[64] = {false};
    const wf_status cst = configure_once(mu, attr_set, [] {
        return cudaFuncSetAttribute(gemm_select_kernel<1, false, true, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_MAX) == cudaSuccess;
    });
    if (cst != WF_OK) return cst;
    GemmParams p = params_for(ws);
    const int num_m = cdiv(P, BM);
    TileGeom tg;
    if (balanced_tiles(V, num_sms(), &tg)) {
        p.num_n = tg.num_n;
        p.bn = tg.bn;
        p.nbig = tg.nbig;
    } else {
        p.bn = pick_bn(num_m, V, num_sms());
        p.num_n = p.nbig = cdiv(V, p.bn);
    }
    // draft head: balanced tiles too (the same number for every CTA pair),
    // half of each loaded by either CTA of a pair
    TileGeom tg2;
    if (balanced_tiles(Vd, num_sms(), &tg2)) {
        p.num_n2 = tg2.num_n;
        p.bn2 = tg2.bn;
        p.nbig2 = tg2.nbig;
    } else {
        p.bn2 = BN;
        p.num_n2 = p.nbig2 = cdiv(Vd, BN);
    }
    CUtensorMap ta, tb, tbs, ta2, tb2, tb2s;
    if (!make_map(&ta, hidden, (uint64_t)P, (uint64_t)d, (uint32_t)BM) ||
        !make_map(&tb, W, (uint64_t)V, (uint64_t)d, (uint32_t)(p.bn / 2)) ||
        !make_map(&ta2, x, (uint64_t)B, (uint64_t)d, (uint32_t)BM) ||
        !make_map(&tb2, Wd, (uint64_t)Vd, (uint64_t)d, (uint32_t)(p.bn2 / 2)))
        return WF_ERR_CUDA;
    tbs = tb;
    tb2s = tb2;
    if (p.nbig < p.num_n && !make_map(&tbs, W, (uint64_t)V, (uint64_t)d, (uint32_t)((p.bn - 16) / 2)))
        return WF_ERR_CUDA;
    if (p.nbig2 < p.num_n2 && !make_map(&tb2s, Wd, (uint64_t)Vd, (uint64_t)d, (uint32_t)((p.bn2 - 16) / 2)))
        return WF_ERR_CUDA;
    p.M_rows = P;
    p.N_w = V;
    p.num_m = num_m;
    p.idesc = umma_idesc_bf16(2 * BM, p.bn);
    p.idesc_s = p.nbig < p.num_n ? umma_idesc_bf16(2 * BM, p.bn - 16) : p.idesc;
    p.idesc2 = umma_idesc_bf16(2 * BM, p.bn2);
    p.idesc2_s = p.nbig2 < p.num_n2 ? umma_idesc_bf16(2 * BM, p.bn2 - 16) : p.idesc2;
    p.num_k = cdiv(d, BK);
    p.weight_evict_first = 1;
    // activation groups as in the plain paired sweep (launch_select)
    const int num_mt = cdiv(num_m, 2);
    const long per_mt = 2L * BM * d * 2;
    const int most = (int)(PAIR_GROUP_BYTES / per_mt) > 0 ? (int)(PAIR_GROUP_BYTES / per_mt) : 1;
    p.group = cdiv(num_mt, cdiv(num_mt, most));
    p.a_bytes = p.a_bytes2 = BM * BK * 2;
    p.ids = ids;
    p.maxlogit = maxlogit;
    p.k = k;
    p.cand = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ws) + cand_off);
    p.lsep = lsep_off ? reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(ws) + lsep_off) : nullptr;
    p.M_rows2 = B;
    p.N_w2 = Vd;
    p.timeout_ns = wait_timeout_ns();
    *num_n2_out = p.num_n2;
    const int smem = set_ring(p, 0, true);
    const int pairs = num_mt * p.num_n + p.num_n2;
    const int slots = pair_slots<1, true>(smem);
    const int grid = 2 * (pairs < slots ? pairs : slots);
    return launch_cluster(gemm_select_kernel<1, false, true, true>, dim3(grid), dim3(GEMM_THREADS), smem, s, 2u, ta,
                          tb, ta2, tb2, tbs, tb2s, p);
}

// Target LM head (argmax over P <= BM rows) and draft head (candidate lists of
// the top k over B <= BM rows) in one persistent sweep of W then Wd (more rows:
// launch_lmhead_draft_pair).  The
// candidate lists are merged by launch_topk_merge over the draft-head tile
// count this returns in *num_n2_out.
wf_status launch_lmhead_draft(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                              float* maxlogit, const uint16_t* x, const uint16_t* Wd, int B, int Vd, int k, void* ws,
                              size_t cand_off, size_t lsep_off, int* num_n2_out, cudaStream_t s, float* H, float tau,
                              size_t ent_off, int* defer_slots) {
    if (P > BM) {
        if (B > 2 * BM || H || defer_slots) return WF_ERR_UNSUPPORTED;
        return launch_lmhead_draft_pair(hidden, W, P, d, V, ids, maxlogit, x, Wd, B, Vd, k, ws, cand_off, lsep_off,
                                        num_n2_out, s);
    }
    if (B > BM) return WF_ERR_UNSUPPORTED;
    static std::mutex mu;
    static bool attr_set[64] = {false};
    const wf_status cst = configure_once(mu, attr_set, [] {
        return cudaFuncSetAttribute(gemm_select_kernel<1, false, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    GEMM_SMEM_MAX) == cudaSuccess &&
               cudaFuncSetAttribute(gemm_select_kernel<1, true, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    GEMM_SMEM_MAX) == cudaSuccess;
    });
    if (cst != WF_OK) return cst;
    const int sms = num_sms();
    GemmParams p = params_for(ws);
    // both matrices in balanced tiles (every CTA sweeps the same rows of each),
    // else one uniform tile height over both
    TileGeom g1, g2;
    if (balanced_tiles(V, sms, &g1) && balanced_tiles(Vd, sms, &g2)) {
        p.num_n = g1.num_n;
        p.bn = g1.bn;
        p.nbig = g1.nbig;
        p.num_n2 = g2.num_n;
        p.bn2 = g2.bn;
        p.nbig2 = g2.nbig;
    } else {
        p.bn = p.bn2 = pick_bn(1, V, sms, Vd);
        p.num_n = p.nbig = cdiv(V, p.bn);
        p.num_n2 = p.nbig2 = cdiv(Vd, p.bn);
    }
    const int a_rows = (P + 7) / 8 * 8, a_rows2 = (B + 7) / 8 * 8;
    CUtensorMap ta, tb, ta2, tb2, tbs, tb2s;
    if (!make_map(&ta, hidden, (uint64_t)P, (uint64_t)d, (uint32_t)a_rows) ||
        !make_map(&tb, W, (uint64_t)V, (uint64_t)d, (uint32_t)p.bn) ||
        !make_map(&ta2, x, (uint64_t)B, (uint64_t)d, (uint32_t)a_rows2) ||
        !make_map(&tb2, Wd, (uint64_t)Vd, (uint64_t)d, (uint32_t)p.bn2))
        return WF_ERR_CUDA;
    tbs = tb;
    tb2s = tb2;
    if (p.nbig < p.num_n && !make_map(&tbs, W, (uint64_t)V, (uint64_t)d, (uint32_t)(p.bn - 16))) return WF_ERR_CUDA;
    if (p.nbig2 < p.num_n2 && !make_map(&tb2s, Wd, (uint64_t)Vd, (uint64_t)d, (uint32_t)(p.bn2 - 16)))
        return WF_ERR_CUDA;
    p.M_rows = P;
    p.N_w = V;
    p.num_m = 1;
    p.idesc = umma_idesc_bf16(BM, p.bn);
    p.idesc_s = p.nbig < p.num_n ? umma_idesc_bf16(BM, p.bn - 16) : p.idesc;
    p.idesc2 = umma_idesc_bf16(BM, p.bn2);
    p.idesc2_s = p.nbig2 < p.num_n2 ? umma_idesc_bf16(BM, p.bn2 - 16) : p.idesc2;
    p.num_k = cdiv(d, BK);
    p.weight_evict_first = 1;
    p.group = 1;
    p.a_bytes = a_rows * BK * 2;
    p.ids = ids;
    p.maxlogit = maxlogit;
    p.k = k;
    p.cand = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ws) + cand_off);
    p.lsep = lsep_off ? reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(ws) + lsep_off) : nullptr;
    p.M_rows2 = B;
    p.N_w2 = Vd;
    p.a_bytes2 = a_rows2 * BK * 2;
    p.timeout_ns = wait_timeout_ns();
    const int tiles = p.num_n + p.num_n2;
    *num_n2_out = p.num_n2;
    const int smem = set_ring(p, a_rows > a_rows2 ? a_rows : a_rows2);
    int grid = tiles < sms ? tiles : sms;
    if (H || defer_slots) {   // the target head's entropy statistics as well (WhiFlash-Entropy)
        p.ent = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(ws) + ent_off);
        p.H = H;
        p.ent_defer = defer_slots != nullptr;
        p.route = nullptr;
        p.tau = tau;
        p.src_rows = nullptr;
        p.src_P = 0;
        if (grid > ENT_MAX_SLOTS) grid = ENT_MAX_SLOTS;
        if (defer_slots) *defer_slots = grid;
        return launch(gemm_select_kernel<1, true, true, false>, dim3(grid), dim3(GEMM_THREADS), smem, s, ta, tb, ta2,
                      tb2, tbs, tb2s, p);
    }
    return launch(gemm_select_kernel<1, false, true, false>, dim3(grid), dim3(GEMM_THREADS), smem, s, ta, tb, ta2, tb2,
                  tbs, tb2s, p);
}

// The merge of the per-tile candidate lists of B rows (num_n weight tiles)
// into the top k, mapped through d2t.
MergeArgs merge_args(int B, int Vd, int num_n, int k, const int32_t* d2t, int32_t* draft_ids, int32_t* tids,
                     float* vals, void* ws, size_t cand_off, float* lse, size_t lsep_off) {
    MergeArgs a = {};
    a.cand = reinterpret_cast<const uint64_t*>(reinterpret_cast<uint8_t*>(ws) + cand_off);
    a.lse = lse;
    a.lsep = lse ? reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(ws) + lsep_off) : nullptr;
    a.B = B;
    a.num_m = cdiv(B, BM);
    a.num_n = num_n;
    a.k = k;
    a.d2t = d2t;
    a.Vd = Vd;
    a.draft_ids = draft_ids;
    a.tids = tids;
    a.vals = vals;
    return a;
}

wf_status launch_topk_merge(const MergeArgs& a, void* ws, cudaStream_t s) {
    if (a.B == 0) return WF_OK;
    return launch(topk_merge_kernel, dim3(a.B), dim3(MERGE_THREADS), 0, s, a, reinterpret_cast<Control*>(ws));
}

}  // namespace wf
