// EAGLE-3 draft-tree construction (the context-aware dynamic tree; WhiFlash
// paper App. A / Table 7: depth 8, top-k 10, 60 draft tokens; EAGLE3 model
// card "Factors").  Given, for every expansion step and frontier slot, the
// drafter's top-k children (target ids and draft log-probabilities), it keeps
// the k best children of each step (cumulative score = parent's + own
// log-probability) as the next frontier, and returns the N best of every child
// created as a parent-array tree listed depth by depth - the tree the next
// verification round checks.
//
// One warp per sequence; the candidate pool lives in shared memory.  Scores
// are summed in fp32 in creation order; every ranking is a warp-wide max over
// packed (order-preserving score, ~creation index) keys, so ties go to the
// node created first.
#include "wf_internal.cuh"

namespace wf {

constexpr int TREE_WARPS = 2;

struct TreePool {   // per warp, in dynamic shared memory
    float* score;
    int32_t* token;
    int16_t* parent;
    int16_t* new_of;
    int8_t* depth;
    uint8_t* taken;
};

__host__ __device__ constexpr size_t tree_pool_bytes(int pool_n) {
    return align_up((size_t)pool_n * (4 + 4 + 2 + 2 + 1 + 1), 16);
}

__device__ __forceinline__ TreePool tree_pool(uint8_t* base, int pool_n) {
    TreePool t;
    t.score = reinterpret_cast<float*>(base);
    t.token = reinterpret_cast<int32_t*>(base + 4 * (size_t)pool_n);
    t.parent = reinterpret_cast<int16_t*>(base + 8 * (size_t)pool_n);
    t.new_of = reinterpret_cast<int16_t*>(base + 10 * (size_t)pool_n);
    t.depth = reinterpret_cast<int8_t*>(base + 12 * (size_t)pool_n);
    t.taken = reinterpret_cast<uint8_t*>(base + 13 * (size_t)pool_n);
    return t;
}

// Best candidate in [lo, hi) whose mark equals `want` (and, if dd > 0, of that
// depth): warp-wide max of packed keys.  The winner's mark becomes `mark`.
// Returns its pool index, or -1 if there is none.
__device__ __forceinline__ int take_best(const TreePool& t, int lo, int hi, uint8_t want, int dd, uint8_t mark,
                                         int lane) {
    uint64_t best = 0;
    for (int i = lo + lane; i < hi; i += 32)
        if (t.taken[i] == want && (dd <= 0 || t.depth[i] == dd)) {
            const uint64_t key = pack_key(t.score[i], (uint32_t)i);
            best = key > best ? key : best;
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
    }
    if (!best) return -1;
    const int idx = (int)key_id(best);
    __syncwarp();
    if (lane == 0) t.taken[idx] = mark;
    __syncwarp();
    return idx;
}

__global__ void __launch_bounds__(TREE_WARPS * 32)
    build_tree_kernel(const int32_t* __restrict__ tid, const float* __restrict__ lp, int B, int D, int k, int N,
                      int32_t* parent, int32_t* token, float* score, int32_t* depth, Control* ctrl) {
    extern __shared__ uint8_t smem_raw[];
    pdl_wait();
    pdl_trigger();
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * TREE_WARPS + w;
    if (b >= B) return;
    const int pool_n = k + (D - 1) * k * k;
    const TreePool t = tree_pool(smem_raw + (size_t)w * tree_pool_bytes(pool_n), pool_n);
    const int32_t* T = tid + (size_t)b * D * k * k;
    const float* L = lp + (size_t)b * D * k * k;

    // marks: 0 = in the pool, 1 = chosen (frontier step / final tree), 2 = listed
    int frontier = -1;   // lane j < k holds frontier slot j (a pool index)
    int made = 0;
    bool bad = false;
    for (int s = 0; s < D; ++s) {
        const int n_step = (s == 0 ? 1 : k) * k;
        // the children of this step: pool [made, made + n_step)
        for (int i0 = 0; i0 < n_step; i0 += 32) {
            const int i = i0 + lane;
            const int j = i / k;
            const int par = __shfl_sync(0xffffffffu, frontier, j < 32 ? j : 0);
            if (i < n_step) {
                const int c = i - j * k;
                const float l = L[((size_t)s * k + j) * k + c];
                bad |= !(l <= 0.0f);
                const int pidx = s == 0 ? -1 : par;
                t.score[made + i] = (pidx < 0 ? 0.0f : t.score[pidx]) + l;
                t.parent[made + i] = (int16_t)pidx;
                t.token[made + i] = T[((size_t)s * k + j) * k + c];
                t.depth[made + i] = (int8_t)(s + 1);
                t.taken[made + i] = 0;
            }
        }
        __syncwarp();
        // the k best children of this step become the next frontier, in rank order
        int next = -1;
        for (int j = 0; j < k; ++j) {
            const int idx = take_best(t, made, made + n_step, 0, 0, 1, lane);
            if (lane == j) next = idx;
        }
        frontier = next;
        made += n_step;
    }
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) record_error(ctrl, WF_ERR_BAD_DATA, (uint32_t)b);
        for (int i = lane; i < N; i += 32) {
            parent[(size_t)b * N + i] = -1;
            token[(size_t)b * N + i] = -1;
            if (score) score[(size_t)b * N + i] = 0.f;
            if (depth) depth[(size_t)b * N + i] = -1;
        }
        return;
    }
    // the N best of the whole pool ...
    for (int i = lane; i < pool_n; i += 32) {
        t.taken[i] = 0;
        t.new_of[i] = -1;
    }
    __syncwarp();
    for (int r = 0; r < N; ++r) take_best(t, 0, pool_n, 0, 0, 1, lane);
    // ... listed depth by depth, in rank order within a depth
    int n_done = 0;
    for (int dd = 1; dd <= D; ++dd)
        for (;;) {
            const int idx = take_best(t, 0, pool_n, 1, dd, 2, lane);
            if (idx < 0) break;
            if (lane == 0) t.new_of[idx] = (int16_t)n_done;
            ++n_done;
        }
    __syncwarp();
    for (int i = lane; i < pool_n; i += 32) {
        const int o = t.new_of[i];
        if (o >= 0) {
            const int pi = t.parent[i];
            parent[(size_t)b * N + o] = pi < 0 ? -1 : t.new_of[pi];
            token[(size_t)b * N + o] = t.token[i];
            if (score) score[(size_t)b * N + o] = t.score[i];
            if (depth) depth[(size_t)b * N + o] = t.depth[i];
        }
    }
}

size_t build_tree_smem(int D, int k) { return tree_pool_bytes(k + (D - 1) * k * k) * TREE_WARPS; }

wf_status launch_build_tree(const int32_t* tid, const float* lp, int B, int D, int k, int N, int32_t* parent,
                            int32_t* token, float* score, int32_t* depth, void* ws, cudaStream_t s) {
    if (B == 0) return WF_OK;
    const size_t smem = build_tree_smem(D, k);
    static std::mutex mu;
    static bool attr_set[64] = {false};
    const wf_status cst = configure_once(mu, attr_set, [] {
        return cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) ==
               cudaSuccess;
    });
    if (cst != WF_OK) return cst;
    return launch(build_tree_kernel, dim3(cdiv(B, TREE_WARPS)), dim3(TREE_WARPS * 32), smem, s, tid, lp, B, D, k, N,
                  parent, token, score, depth, reinterpret_cast<Control*>(ws));
}

}  // namespace wf
