// The draft head's top-k merge (EAGLE-3 draft head, "top-k" candidates of
// the next-token distribution over the draft vocabulary, mapped to target ids
// through d2t): the per-tile sorted candidate lists of one activation row,
// merged into its k best.  Used by topk_merge_kernel and, inside a round, by
// extra CTAs of the verification launch (the merge depends only on the weight
// sweep, so it runs beside the verification instead of after it).
#pragma once

#include "wf_internal.cuh"

namespace wf {

constexpr int MERGE_THREADS = 128;
// Shared scratch of one merge (8-byte words): a word per warp for the
// block-wide max, then the k winners in order.
constexpr int MERGE_SCRATCH = MERGE_THREADS / 32 + WF_MAX_TOPK;

struct MergeArgs {
    const uint64_t* cand;   // [num_n][num_m * BM][k] packed keys (0 = none), zeroed as read
    int B, num_m, num_n, k;
    const int32_t* d2t;     // [Vd] draft id -> target id
    int Vd;
    int32_t* draft_ids;     // [B, k] or null
    int32_t* tids;          // [B, k] or null
    float* vals;            // [B, k] or null
    float2* lsep;           // [num_n][num_m * BM] per-tile (max, sum e^(logit - max)), zeroed as read; or null
    float* lse;             // [B] log-sum-exp of the row's logits over the draft vocabulary, or null
};

// One CTA (MERGE_THREADS threads) merges row `row`: every thread keeps the
// WF_MAX_TOPK best of its share of the candidate lists, then k rounds of a
// block-wide max pick the winners in order (on chip only); k threads then
// map the winners to target ids and write them, all lookups in flight
// together.  Keys are unique per row (each weight row lives in one tile), so
// exactly one thread owns each winner.  wbest: MERGE_SCRATCH words of shared
// memory.  BATCH candidates of a thread are loaded together: the standalone
// merge (many rows, a CTA each) loads all of them at once, the merge CTAs
// beside the verification keep to a few.
template <int BATCH>
__device__ __forceinline__ void topk_merge_row(const MergeArgs& a, int row, uint64_t* wbest, Control* ctrl) {
    constexpr int KT = WF_MAX_TOPK;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m = row / BM, rit = row % BM;
    const int k = a.k;
    if (a.lsep) {
        // log-sum-exp over the draft vocabulary: every thread folds its tiles'
        // (max, sum) pairs in increasing tile order, then a fixed shuffle tree
        // and the warps in order (the same result on every run)
        float M = -INFINITY, S = 0.f;
        for (int n = threadIdx.x; n < a.num_n; n += MERGE_THREADS) {
            float2* src = a.lsep + ((size_t)n * a.num_m + m) * BM + rit;
            const float2 v = *src;
            *src = make_float2(0.f, 0.f);   // leave the workspace zeroed
            lse_merge(M, S, v.x, v.y);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, M, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, S, off);
            lse_merge(M, S, m2, s2);
        }
        float2* wl = reinterpret_cast<float2*>(wbest);   // MERGE_THREADS / 32 words of 8 bytes
        if (lane == 0) wl[warp] = make_float2(M, S);
        __syncthreads();
        if (threadIdx.x == 0) {
            float Mt = -INFINITY, St = 0.f;
#pragma unroll
            for (int w = 0; w < MERGE_THREADS / 32; ++w) lse_merge(Mt, St, wl[w].x, wl[w].y);
            a.lse[row] = St > 0.f ? Mt + logf(St) : __int_as_float(0x7fc00000);
        }
        __syncthreads();   // wbest is reused below
    }
    uint64_t loc[KT];
#pragma unroll
    for (int j = 0; j < KT; ++j) loc[j] = 0;
    const int total = a.num_n * k;
    for (int base = 0; base < total; base += MERGE_THREADS * BATCH) {
        uint64_t kb[BATCH];
        uint64_t* src[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int idx = base + u * MERGE_THREADS + threadIdx.x;
            const int n = idx / k, j = idx - n * k;
            src[u] = idx < total ? const_cast<uint64_t*>(a.cand) + (((size_t)n * a.num_m + m) * BM + rit) * k + j
                                 : nullptr;
            kb[u] = src[u] ? *src[u] : 0ull;
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u)
            if (src[u]) *src[u] = 0;  // leave the workspace zeroed
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const uint64_t key = kb[u];
            if (key > loc[KT - 1]) {
#pragma unroll
                for (int s = KT - 1; s > 0; --s) {
                    const bool shift = loc[s - 1] < key;
                    const bool land = !shift && loc[s] < key;
                    loc[s] = shift ? loc[s - 1] : (land ? key : loc[s]);
                }
                if (loc[0] < key) loc[0] = key;
            }
        }
    }
    for (int j = 0; j < k; ++j) {
        uint64_t best = loc[0];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o > best ? o : best;
        }
        if (lane == 0) wbest[warp] = best;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < MERGE_THREADS / 32; ++w) best = wbest[w] > best ? wbest[w] : best;
        __syncthreads();   // every thread has read wbest before the next round writes it
        if (loc[0] == best && best != 0) {  // the (unique) owner pops its head
#pragma unroll
            for (int s = 0; s < KT - 1; ++s) loc[s] = loc[s + 1];
            loc[KT - 1] = 0;
        }
        if (threadIdx.x == 0) wbest[MERGE_THREADS / 32 + j] = best;
    }
    __syncthreads();
    if ((int)threadIdx.x < k) {
        const int j = threadIdx.x;
        const uint64_t best = wbest[MERGE_THREADS / 32 + j];
        const size_t o = (size_t)row * k + j;
        int32_t id = -1, tid = -1;
        float v = __int_as_float(0x7fc00000);
        if (best != 0) {
            id = (int32_t)key_id(best);
            v = key_val(best);
            tid = (id >= 0 && id < a.Vd) ? a.d2t[id] : -1;
            if (tid < 0) record_error(ctrl, WF_ERR_BAD_DATA, (uint32_t)row);
        }
        if (a.draft_ids) a.draft_ids[o] = id;
        if (a.tids) a.tids[o] = tid;
        if (a.vals) a.vals[o] = v;
    }
}

}  // namespace wf
