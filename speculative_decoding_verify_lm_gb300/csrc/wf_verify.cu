// Greedy acceptance of drafted DFlash chains and EAGLE-3 trees, one warp per
// sequence (WhiFlash paper Sec. 3.2: the drafted block or tree is verified by
// the target in parallel and decoding resumes from the last accepted token).
//
// Chain: the accepted prefix ends at the first drafted token that differs
// from the target's choice at the row before it - a warp ballot over 32
// drafts at a time.
// Tree: node i is accepted iff its token equals the target's choice at its
// parent's row and every ancestor is accepted.  The warp computes the match
// flag of every node in parallel, then pointer-jumps (each round doubles the
// span of ancestors folded in) to get, per node, the AND over its whole root
// path and its depth; the deepest accepted node (lowest index on a tie) wins
// a warp max over packed (depth, ~index) keys.
#include "wf_internal.cuh"
#include "wf_merge.cuh"

namespace wf {

constexpr int VERIFY_WARPS = 4;
constexpr int NODES_PER_LANE = WF_MAX_SEQ_NODES / 32;

__global__ void __launch_bounds__(VERIFY_WARPS * 32)
    verify_kernel(const int32_t* __restrict__ g, const int32_t* __restrict__ tok, const int32_t* __restrict__ parent,
                  const int32_t* __restrict__ kind, int default_kind, const int32_t* __restrict__ pos_off,
                  const int32_t* __restrict__ node_off, int B, int P, int path_stride, int32_t* n_accept,
                  int32_t* bonus, int32_t* last_pos, int32_t* path, RoutePick pick, int early_inputs,
                  MergeArgs mg, int nverify, Control* ctrl) {
    __shared__ int16_t s_par[VERIFY_WARPS][WF_MAX_SEQ_NODES];
    __shared__ int16_t s_anc[VERIFY_WARPS][WF_MAX_SEQ_NODES];
    __shared__ int16_t s_dist[VERIFY_WARPS][WF_MAX_SEQ_NODES];
    __shared__ uint8_t s_ok[VERIFY_WARPS][WF_MAX_SEQ_NODES];
    __shared__ int32_t s_g[VERIFY_WARPS][WF_MAX_SEQ_NODES + 1];

    // CTAs past the verification ones merge the draft head's candidate lists
    // (one row each): they depend on the weight sweep only, like verification
    if ((int)blockIdx.x >= nverify) {
        __shared__ uint64_t s_wbest[MERGE_SCRATCH];
        pdl_wait();
        pdl_trigger();
        topk_merge_row<4>(mg, (int)blockIdx.x - nverify, s_wbest, ctrl);
        return;
    }
    const unsigned FULL = 0xffffffffu;
    const int w = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * VERIFY_WARPS + w;
    const bool live = b < B;

    // ---- inside a round the predecessor is the round's LM head (or the router
    // beside it), which started only after everything before the round had
    // finished: the round's own inputs (offsets, drafts, parents) are read
    // while it is still running.  A call of its own reads them after the wait.
    if (!early_inputs) pdl_wait();
    int r0 = 0, N = 0, kd = default_kind;
    bool shape_ok = false;
    int tk[NODES_PER_LANE], pa[NODES_PER_LANE];
    if (live) {
        r0 = pos_off[b];
        const int r1 = pos_off[b + 1];
        const int n0 = node_off[b];
        N = node_off[b + 1] - n0;
        shape_ok = r0 >= 0 && r1 > r0 && (P < 0 || r1 <= P) && n0 >= 0 && N >= 0 && N == r1 - r0 - 1 &&
                   N <= WF_MAX_SEQ_NODES;
        kd = kind ? kind[b] : default_kind;
#pragma unroll
        for (int s = 0; s < NODES_PER_LANE; ++s) {
            const int i = lane + 32 * s;
            const bool in = shape_ok && i < N;
            tk[s] = in ? tok[n0 + i] : 0;
            pa[s] = (in && kd != 0 && parent) ? parent[n0 + i] : -1;
        }
    }
    if (early_inputs) pdl_wait();   // the target choices g come from the kernel before this one
    pdl_trigger();
    if (!live) return;

    auto fail = [&]() {   // warp-uniform
        if (lane == 0) {
            record_error(ctrl, WF_ERR_BAD_DATA, (uint32_t)b);
            n_accept[b] = -1;
            bonus[b] = -1;
            last_pos[b] = -1;
        }
        pick.publish(b, -1, lane);
        if (path)
            for (int j = lane; j < path_stride; j += 32) path[(size_t)b * path_stride + j] = -1;
    };
    if (!shape_ok || (kd != 0 && !parent)) {
        fail();
        return;
    }
    int32_t* gs = s_g[w];   // target choice at each of this sequence's rows
    for (int r = lane; r <= N; r += 32) gs[r] = g[r0 + r];
    __syncwarp();

    if (kd == 0) {
        // ---------------------------------------------------------------- chain
        int n = N;
#pragma unroll
        for (int s = 0; s < NODES_PER_LANE; ++s) {
            const int base = 32 * s;
            if (base >= N) break;
            const int j = base + lane;
            const unsigned mask = __ballot_sync(FULL, j < N && tk[s] != gs[j]);
            if (mask) {
                n = base + __ffs(mask) - 1;
                break;
            }
        }
        if (lane == 0) {
            n_accept[b] = n;
            last_pos[b] = r0 + n;
            bonus[b] = gs[n];
        }
        pick.publish(b, r0 + n, lane);
        if (path)
            for (int j = lane; j < path_stride; j += 32) path[(size_t)b * path_stride + j] = j < n ? j : -1;
        return;
    }

    // -------------------------------------------------------------------- tree
    int16_t* par = s_par[w];
    int16_t* anc = s_anc[w];
    int16_t* dist = s_dist[w];
    uint8_t* okf = s_ok[w];
    bool bad = false;
#pragma unroll
    for (int s = 0; s < NODES_PER_LANE; ++s) {
        const int i = lane + 32 * s;
        if (i < N) {
            const int pi = pa[s];
            const bool pbad = pi < -1 || pi >= i;
            bad |= pbad;
            par[i] = (int16_t)(pbad ? -1 : pi);
            anc[i] = par[i];
            dist[i] = 1;
            okf[i] = (uint8_t)(!pbad && tk[s] == gs[pi < 0 ? 0 : 1 + pi]);
        }
    }
    if (__any_sync(FULL, bad)) {
        fail();
        return;
    }
    __syncwarp();
    // pointer jumping: invariant - okf[i] = AND of the match flags of the dist[i]
    // nodes from i up to (excluding) anc[i]
    for (int span = 1; span < N; span <<= 1) {
        int16_t na[NODES_PER_LANE], nd[NODES_PER_LANE];
        uint8_t no[NODES_PER_LANE];
        bool more = false;
#pragma unroll
        for (int s = 0; s < NODES_PER_LANE; ++s) {
            const int i = lane + 32 * s;
            if (i < N) {
                const int a = anc[i];
                if (a >= 0) {
                    na[s] = anc[a];
                    nd[s] = (int16_t)(dist[i] + dist[a]);
                    no[s] = okf[i] & okf[a];
                    more = true;
                } else {
                    na[s] = -1;
                    nd[s] = dist[i];
                    no[s] = okf[i];
                }
            }
        }
        if (!__any_sync(FULL, more)) break;
        __syncwarp();
#pragma unroll
        for (int s = 0; s < NODES_PER_LANE; ++s) {
            const int i = lane + 32 * s;
            if (i < N) {
                anc[i] = na[s];
                dist[i] = nd[s];
                okf[i] = no[s];
            }
        }
        __syncwarp();
    }
    // deepest accepted node, lowest index on equal depth
    uint32_t best = 0;
    for (int i = lane; i < N; i += 32)
        if (okf[i]) {
            const uint32_t key = ((uint32_t)dist[i] << 16) | (uint32_t)(0xFFFF - i);
            best = key > best ? key : best;
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const uint32_t o = __shfl_xor_sync(FULL, best, off);
        best = o > best ? o : best;
    }
    const int n = (int)(best >> 16);
    const int node = best ? 0xFFFF - (int)(best & 0xFFFF) : -1;
    if (path) {
        for (int j = lane; j < path_stride; j += 32) path[(size_t)b * path_stride + j] = -1;
        __syncwarp();
        if (lane == 0)
            for (int i = node, dep = n; i >= 0; i = par[i], --dep)
                if (dep - 1 < path_stride) path[(size_t)b * path_stride + dep - 1] = i;
    }
    if (lane == 0) {
        n_accept[b] = n;
        last_pos[b] = r0 + 1 + node;   // the root row when node = -1
        bonus[b] = gs[1 + node];
    }
    pick.publish(b, r0 + 1 + node, lane);
}

wf_status launch_verify(const int32_t* g, const int32_t* tok, const int32_t* parent, const int32_t* kind,
                        int default_kind, const int32_t* pos_off, const int32_t* node_off, int B, int P,
                        int path_stride, int32_t* n_accept, int32_t* bonus, int32_t* last_pos, int32_t* path,
                        void* ws, cudaStream_t s, RoutePick pick, bool early_inputs, const MergeArgs* merge) {
    static_assert(MERGE_THREADS == VERIFY_WARPS * 32, "merge CTAs share the verification launch's block size");
    const int nverify = cdiv(B, VERIFY_WARPS);
    const int nmerge = merge ? merge->B : 0;
    if (nverify + nmerge == 0) return WF_OK;
    return launch(verify_kernel, dim3(nverify + nmerge), dim3(VERIFY_WARPS * 32), 0, s, g, tok, parent, kind,
                  default_kind, pos_off, node_off, B, P, path_stride, n_accept, bonus, last_pos, path, pick,
                  (int)early_inputs, merge ? *merge : MergeArgs{}, nverify, reinterpret_cast<Control*>(ws));
}

}  // namespace wf

namespace wf {

// Exercises the bounded-wait path every pipelined kernel uses: one thread
// waits on an mbarrier that nothing arrives on, gives up after timeout_ns and
// records WF_ERR_TIMEOUT in the workspace's error word.
__global__ void bounded_wait_probe_kernel(uint64_t timeout_ns, Control* ctrl) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        if (!mbar_wait(&bar, 0, timeout_ns, nullptr)) record_error(ctrl, WF_ERR_TIMEOUT, 0xFFFFu);
    }
}

wf_status launch_wait_probe(uint64_t timeout_ns, void* ws, cudaStream_t s) {
    bounded_wait_probe_kernel<<<1, 32, 0, s>>>(timeout_ns, reinterpret_cast<Control*>(ws));
    return cudaGetLastError() == cudaSuccess ? WF_OK : WF_ERR_CUDA;
}

}  // namespace wf

namespace wf {

// Rows kept after a round (the committed positions: the root row and the rows
// of the accepted path) and their packed offsets, one CTA: a block-wide
// exclusive scan of n_accept + 1 over the sequences, 1024 at a time.
__global__ void __launch_bounds__(1024)
    accepted_rows_kernel(const int32_t* __restrict__ n_accept, const int32_t* __restrict__ path, int path_stride,
                         const int32_t* __restrict__ pos_off, int B, int32_t* acc_rows, int32_t* acc_off) {
    __shared__ int32_t warp_sum[32];
    __shared__ int32_t carry;
    pdl_wait();   // n_accept / path come from the acceptance step
    pdl_trigger();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        carry = 0;
        acc_off[0] = 0;
    }
    __syncthreads();
    for (int b0 = 0; b0 < B; b0 += blockDim.x) {
        const int b = b0 + threadIdx.x;
        int cnt = 0;
        if (b < B) {
            // n_accept beyond the path's columns is taken as the columns; -1 (a
            // sequence with bad data) keeps no row
            const int n = max(-1, min(n_accept[b], path_stride));
            cnt = n + 1;
            int32_t* out = acc_rows + (size_t)b * (path_stride + 1);
            out[0] = pos_off[b];
            for (int j = 1; j <= path_stride; ++j)
                out[j] = j <= n ? pos_off[b] + 1 + path[(size_t)b * path_stride + j - 1] : -1;
        }
        // inclusive scan of cnt across the block
        int v = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += o;
        }
        if (lane == 31) warp_sum[w] = v;
        __syncthreads();
        if (w == 0) {
            int s = lane < (int)(blockDim.x >> 5) ? warp_sum[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += o;
            }
            warp_sum[lane] = s;
        }
        __syncthreads();
        const int incl = v + (w > 0 ? warp_sum[w - 1] : 0) + carry;
        if (b < B) acc_off[b + 1] = incl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = incl;
        __syncthreads();
    }
}

// hidden_out[acc_off[b] + j] = hidden[acc_rows[b][j]] for the kept rows of sequence b.
__global__ void __launch_bounds__(128)
    gather_kept_kernel(const uint16_t* __restrict__ hidden, int d, const int32_t* __restrict__ acc_rows,
                       const int32_t* __restrict__ acc_off, int path_stride, uint16_t* __restrict__ hidden_out) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int first = acc_off[b], cnt = acc_off[b + 1] - first;
    const int chunks = d >> 3;
    for (int j = 0; j < cnt && j <= path_stride; ++j) {
        const int r = acc_rows[(size_t)b * (path_stride + 1) + j];
        const uint4* src = reinterpret_cast<const uint4*>(hidden + (size_t)r * d);
        uint4* dst = reinterpret_cast<uint4*>(hidden_out + (size_t)(first + j) * d);
        for (int c = threadIdx.x; c < chunks; c += blockDim.x) dst[c] = src[c];
    }
}

wf_status launch_accepted_rows(const int32_t* n_accept, const int32_t* path, int path_stride, const int32_t* pos_off,
                               int B, int32_t* acc_rows, int32_t* acc_off, const uint16_t* hidden, int d,
                               uint16_t* hidden_out, cudaStream_t s) {
    if (B == 0) return WF_OK;
    wf_status st = launch(accepted_rows_kernel, dim3(1), dim3(1024), 0, s, n_accept, path, path_stride, pos_off, B,
                          acc_rows, acc_off);
    if (st != WF_OK || !hidden_out) return st;
    return launch(gather_kept_kernel, dim3(B), dim3(128), 0, s, hidden, d, (const int32_t*)acc_rows,
                  (const int32_t*)acc_off, path_stride, hidden_out);
}

}  // namespace wf
