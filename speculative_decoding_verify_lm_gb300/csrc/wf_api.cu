// C ABI entry points: host-side validation, workspace layout and the
// stream-ordered composition of one verify-and-route round.
#include <atomic>
#include <initializer_list>
#include <mutex>

#include "wf_internal.cuh"
#include "wf_merge.cuh"

namespace wf {

wf_status launch_lmhead_argmax(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                               float* maxlogit, void* ws, cudaStream_t s);
wf_status launch_draft_topk(const uint16_t* x, const uint16_t* Wd, const int32_t* d2t, int B, int d, int Vd, int k,
                            int32_t* draft_ids, int32_t* tids, float* vals, float* lse, void* ws, size_t cand_off,
                            size_t lsep_off, cudaStream_t s);
wf_status launch_verify(const int32_t* g, const int32_t* tok, const int32_t* parent, const int32_t* kind,
                        int default_kind, const int32_t* pos_off, const int32_t* node_off, int B, int P,
                        int path_stride, int32_t* n_accept, int32_t* bonus, int32_t* last_pos, int32_t* path,
                        void* ws, cudaStream_t s, RoutePick pick, bool early_inputs, const MergeArgs* merge = nullptr);
wf_status launch_router(const uint16_t* hidden, const int32_t* rows, int B, int d, int m, int P, const float* W1,
                        const float* b1, const float* w2, float b2, float tau, float* delta_al, int32_t* route,
                        void* ws, size_t part_off, cudaStream_t s);

wf_status launch_wait_probe(uint64_t timeout_ns, void* ws, cudaStream_t s);
wf_status launch_lmhead_entropy(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                                float* maxlogit, float* H, int32_t* route, float tau, const int32_t* src_rows,
                                int src_P, void* ws, size_t ent_off, cudaStream_t s, int* defer_slots = nullptr);
wf_status launch_build_tree(const int32_t* tid, const float* lp, int B, int D, int k, int N, int32_t* parent,
                            int32_t* token, float* score, int32_t* depth, void* ws, cudaStream_t s);
wf_status launch_accepted_rows(const int32_t* n_accept, const int32_t* path, int path_stride, const int32_t* pos_off,
                               int B, int32_t* acc_rows, int32_t* acc_off, const uint16_t* hidden, int d,
                               uint16_t* hidden_out, cudaStream_t s);
wf_status launch_gather_rows(const uint16_t* hidden, int P, int d, const int32_t* rows, int B, uint16_t* out,
                             void* ws, cudaStream_t s);
wf_status launch_lmhead_draft(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                              float* maxlogit, const uint16_t* x, const uint16_t* Wd, int B, int Vd, int k, void* ws,
                              size_t cand_off, size_t lsep_off, int* num_n2_out, cudaStream_t s, float* H = nullptr,
                              float tau = 0.f, size_t ent_off = 0, int* defer_slots = nullptr);
MergeArgs merge_args(int B, int Vd, int num_n, int k, const int32_t* d2t, int32_t* draft_ids, int32_t* tids,
                     float* vals, void* ws, size_t cand_off, float* lse = nullptr, size_t lsep_off = 0);
wf_status launch_topk_merge(const MergeArgs& a, void* ws, cudaStream_t s);
wf_status launch_catchup(const wf_catchup_args* a, void* ws, bool with_final, cudaStream_t s);
size_t catchup_workspace_bytes(int B, int N, int din, int H, int G, int D);
size_t catchup_attend_smem(int H, int G, int D);
wf_status noalloc_lmhead_argmax(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                                float* maxlogit, cudaStream_t s);
wf_status noalloc_read_device_error(int* code, int* info, int clear, cudaStream_t s);

static std::atomic<uint64_t> g_timeout_ns{2000000000ull};
uint64_t wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

static int g_sms[64];
static signed char g_dev_ok[64];  // 0 unknown, 1 sm_103, -1 other

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) return 148;
    if (!g_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 148;
    }
    return g_sms[dev];
}

// The kernels are built for sm_103a only (tcgen05, TMA).
static wf_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WF_ERR_CUDA;
    if (dev < 64 && g_dev_ok[dev]) return g_dev_ok[dev] > 0 ? WF_OK : WF_ERR_UNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return WF_ERR_CUDA;
    const bool ok = major == 10 && minor == 3;
    if (dev < 64) g_dev_ok[dev] = ok ? 1 : -1;
    return ok ? WF_OK : WF_ERR_UNSUPPORTED;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A buffer the kernels read with the tensor-memory accelerator must be memory
// of the current device itself (device or managed memory): a host pointer, or
// another GPU's memory reached through a peer mapping, is refused before any
// tensor map is built or anything enqueued.
static bool local_device_memory(const void* p) {
    if (!p) return true;   // optional operand not given
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();   // clear the error the failed query recorded
        return false;
    }
    if (at.type == cudaMemoryTypeManaged) return true;
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

static wf_status check_local(std::initializer_list<const void*> ptrs) {
    for (const void* p : ptrs)
        if (!local_device_memory(p)) return WF_ERR_INVALID_ARG;
    return WF_OK;
}

static wf_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return WF_ERR_WORKSPACE;
    return ws_bytes >= need ? WF_OK : WF_ERR_WORKSPACE;
}

static bool bad_gemm_shape(int rows, int d, int n) {
    return rows < 1 || n < 1 || d < 8 || d % 8 != 0 || d > 16384;
}

#define WF_TRY(x)                        \
    do {                                 \
        const wf_status _st = (x);       \
        if (_st != WF_OK) return _st;    \
    } while (0)

}  // namespace wf

using namespace wf;

extern "C" {

const char* wf_status_string(int status) {
    switch (status) {
        case WF_OK: return "WF_OK";
        case WF_ERR_INVALID_ARG: return "WF_ERR_INVALID_ARG: invalid argument";
        case WF_ERR_WORKSPACE: return "WF_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case WF_ERR_CUDA: return "WF_ERR_CUDA: CUDA runtime error";
        case WF_ERR_UNSUPPORTED: return "WF_ERR_UNSUPPORTED: needs an sm_103 (GB300) device";
        case WF_ERR_BAD_DATA: return "WF_ERR_BAD_DATA: malformed tree, offsets or id map";
        case WF_ERR_TIMEOUT: return "WF_ERR_TIMEOUT: a bounded device wait gave up";
        default: return "unknown wf_status";
    }
}

int wf_version(void) { return 100; }

size_t wf_workspace_bytes(int P, int B, int d, int m, int Vd, int k) { return layout(P, B, d, m, Vd, k).total; }

void wf_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 2000000000ull); }

wf_status wf_workspace_init(void* ws, size_t ws_bytes, wf_stream_t stream) {
    if (!ws || ws_bytes < sizeof(Control)) return WF_ERR_WORKSPACE;
    return cudaMemsetAsync(ws, 0, ws_bytes, stream) == cudaSuccess ? WF_OK : WF_ERR_CUDA;
}

wf_status wf_read_device_error(void* ws, int* code, int* info, int clear, wf_stream_t stream) {
    if (!ws || !code) return WF_ERR_INVALID_ARG;
    uint32_t h[2] = {0, 0};
    if (cudaMemcpyAsync(h, ws, sizeof h, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return WF_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return WF_ERR_CUDA;
    *code = (int)h[0];
    if (info) *info = (int)h[1];
    if (clear) {
        if (cudaMemsetAsync(ws, 0, sizeof h, stream) != cudaSuccess) return WF_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return WF_ERR_CUDA;
    }
    return WF_OK;
}

wf_status wf_probe_bounded_wait(uint64_t timeout_ns, void* ws, size_t ws_bytes, wf_stream_t stream) {
    if (timeout_ns > 10000000000ull) return WF_ERR_INVALID_ARG;
    WF_TRY(check_ws(ws, ws_bytes, sizeof(Control)));
    WF_TRY(check_device());
    return launch_wait_probe(timeout_ns, ws, stream);
}

wf_status wf_lmhead_argmax(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                           float* maxlogit, void* ws, size_t ws_bytes, wf_stream_t stream) {
    if (!hidden || !W || !ids || bad_gemm_shape(P, d, V)) return WF_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(W)) return WF_ERR_INVALID_ARG;
    WF_TRY(check_ws(ws, ws_bytes, layout(P, 0, d, 0, 0, 0).cand));   // control block and keys
    WF_TRY(check_device());
    WF_TRY(check_local({hidden, W}));
    return launch_lmhead_argmax(hidden, W, P, d, V, ids, maxlogit, ws, stream);
}

wf_status wf_lmhead_argmax_noalloc(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                                   float* maxlogit, wf_stream_t stream) {
    if (!hidden || !W || !ids || bad_gemm_shape(P, d, V) || P > WF_NOALLOC_MAX_ROWS) return WF_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(W)) return WF_ERR_INVALID_ARG;
    WF_TRY(check_device());
    WF_TRY(check_local({hidden, W}));
    return noalloc_lmhead_argmax(hidden, W, P, d, V, ids, maxlogit, stream);
}

wf_status wf_noalloc_read_device_error(int* code, int* info, int clear, wf_stream_t stream) {
    if (!code) return WF_ERR_INVALID_ARG;
    WF_TRY(check_device());
    return noalloc_read_device_error(code, info, clear, stream);
}

wf_status wf_lmhead_entropy(const uint16_t* hidden, int P, int d, const int32_t* rows, int B, const uint16_t* W,
                            int V, float tau, float* H, int32_t* route, void* ws, size_t ws_bytes,
                            wf_stream_t stream) {
    if (!hidden || !W || !H || bad_gemm_shape(P, d, V) || B < 1 || B > ENT_MAX_ROWS) return WF_ERR_INVALID_ARG;
    if (!rows && B > P) return WF_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(W)) return WF_ERR_INVALID_ARG;
    const Layout L = layout(0, B, d, 0, 0, 0);
    WF_TRY(check_ws(ws, ws_bytes, rows ? L.total : L.gath));   // the gather area only when rows are given
    WF_TRY(check_device());
    WF_TRY(check_local({hidden, W, rows ? ws : nullptr}));
    const uint16_t* act = hidden;
    if (rows) {
        uint16_t* gath = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(ws) + L.gath);
        WF_TRY(launch_gather_rows(hidden, P, d, rows, B, gath, ws, stream));
        act = gath;
    }
    return launch_lmhead_entropy(act, W, B, d, V, nullptr, nullptr, H, route, tau, rows, P, ws, L.ent, stream);
}

wf_status wf_build_tree(const int32_t* tid, const float* lp, int B, int D, int k, int N, int32_t* parent,
                        int32_t* token, float* score, int32_t* depth, void* ws, size_t ws_bytes,
                        wf_stream_t stream) {
    if (!tid || !lp || !parent || !token || B < 0 || k < 1 || k > 16 || D < 1 || D > 16) return WF_ERR_INVALID_ARG;
    if (N < 1 || N > k + (D - 1) * k * k) return WF_ERR_INVALID_ARG;
    WF_TRY(check_ws(ws, ws_bytes, sizeof(Control)));
    WF_TRY(check_device());
    return launch_build_tree(tid, lp, B, D, k, N, parent, token, score, depth, ws, stream);
}

wf_status wf_accepted_rows(const int32_t* n_accept, const int32_t* path, int path_stride, const int32_t* pos_off,
                           int B, int32_t* acc_rows, int32_t* acc_off, const uint16_t* hidden, int d,
                           uint16_t* hidden_out, wf_stream_t stream) {
    if (B < 0 || path_stride < 0 || !n_accept || !pos_off || !acc_rows || !acc_off) return WF_ERR_INVALID_ARG;
    if (path_stride > 0 && !path) return WF_ERR_INVALID_ARG;
    if ((hidden == nullptr) != (hidden_out == nullptr)) return WF_ERR_INVALID_ARG;
    if (hidden && (d < 8 || d % 8 != 0 || !aligned16(hidden) || !aligned16(hidden_out))) return WF_ERR_INVALID_ARG;
    WF_TRY(check_device());
    return launch_accepted_rows(n_accept, path, path_stride, pos_off, B, acc_rows, acc_off, hidden, d, hidden_out,
                                stream);
}

wf_status wf_verify_chain(const int32_t* g, const int32_t* draft, const int32_t* pos_off, const int32_t* node_off,
                          int B, int path_stride, int32_t* n_accept, int32_t* bonus, int32_t* last_pos,
                          int32_t* path, void* ws, size_t ws_bytes, wf_stream_t stream) {
    if (B < 0 || path_stride < 0 || (path_stride > 0 && !path)) return WF_ERR_INVALID_ARG;
    if (!g || !draft || !pos_off || !node_off || !n_accept || !bonus || !last_pos) return WF_ERR_INVALID_ARG;
    WF_TRY(check_ws(ws, ws_bytes, sizeof(Control)));
    WF_TRY(check_device());
    return launch_verify(g, draft, nullptr, nullptr, 0, pos_off, node_off, B, -1, path ? path_stride : 0,
                         n_accept, bonus, last_pos, path, ws, stream, RoutePick{}, false);
}

wf_status wf_verify_tree(const int32_t* g, const int32_t* tok, const int32_t* parent, const int32_t* node_off,
                         const int32_t* pos_off, int B, int path_stride, int32_t* n_accept, int32_t* bonus,
                         int32_t* last_pos, int32_t* path, void* ws, size_t ws_bytes, wf_stream_t stream) {
    if (B < 0 || path_stride < 0 || (path_stride > 0 && !path)) return WF_ERR_INVALID_ARG;
    if (!g || !tok || !parent || !pos_off || !node_off || !n_accept || !bonus || !last_pos)
        return WF_ERR_INVALID_ARG;
    WF_TRY(check_ws(ws, ws_bytes, sizeof(Control)));
    WF_TRY(check_device());
    return launch_verify(g, tok, parent, nullptr, 1, pos_off, node_off, B, -1, path ? path_stride : 0, n_accept,
                         bonus, last_pos, path, ws, stream, RoutePick{}, false);
}

wf_status wf_router_mlp(const uint16_t* hidden, const int32_t* rows, int B, int d, int m, const float* W1,
                        const float* b1, const float* w2, float b2, float tau, float* delta_al, int32_t* route,
                        void* ws, size_t ws_bytes, wf_stream_t stream) {
    if (B < 0 || d < 8 || d % 8 != 0 || m < 1 || m > ROUTER_MAX_WIDTH) return WF_ERR_INVALID_ARG;
    if (!hidden || !rows || !W1 || !b1 || !w2 || (!delta_al && !route)) return WF_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(W1)) return WF_ERR_INVALID_ARG;
    const Layout L = layout(0, B, d, m, 0, 0);
    WF_TRY(check_ws(ws, ws_bytes, L.dall));   // up to the end of the router partials
    WF_TRY(check_device());
    return launch_router(hidden, rows, B, d, m, -1, W1, b1, w2, b2, tau, delta_al, route, ws, L.part, stream);
}

wf_status wf_draft_topk(const uint16_t* x, const uint16_t* Wd, const int32_t* d2t, int B, int d, int Vd, int k,
                        int32_t* draft_ids, int32_t* tids, float* vals, float* lse, void* ws, size_t ws_bytes,
                        wf_stream_t stream) {
    if (!x || !Wd || !d2t || bad_gemm_shape(B, d, Vd)) return WF_ERR_INVALID_ARG;
    if (k < 1 || k > WF_MAX_TOPK || k > Vd || (!draft_ids && !tids && !vals && !lse)) return WF_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wd)) return WF_ERR_INVALID_ARG;
    const Layout L = layout(0, B, d, 0, Vd, k);
    WF_TRY(check_ws(ws, ws_bytes, L.part));   // up to the end of the top-k candidates and their sums
    WF_TRY(check_device());
    WF_TRY(check_local({x, Wd}));
    return launch_draft_topk(x, Wd, d2t, B, d, Vd, k, draft_ids, tids, vals, lse, ws, L.cand, L.lsep, stream);
}

wf_status wf_lmhead_draft_topk(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                               float* maxlogit, const uint16_t* x, const uint16_t* Wd, const int32_t* d2t, int B,
                               int Vd, int k, int32_t* draft_ids, int32_t* tids, float* vals, float* lse, void* ws,
                               size_t ws_bytes, wf_stream_t stream) {
    if (!hidden || !W || !ids || bad_gemm_shape(P, d, V)) return WF_ERR_INVALID_ARG;
    if (!x || !Wd || !d2t || bad_gemm_shape(B, d, Vd)) return WF_ERR_INVALID_ARG;
    if (k < 1 || k > WF_MAX_TOPK || k > Vd || (!draft_ids && !tids && !vals && !lse)) return WF_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(W) || !aligned16(x) || !aligned16(Wd)) return WF_ERR_INVALID_ARG;
    if (P <= BM ? B > BM : B > 2 * BM) return WF_ERR_UNSUPPORTED;
    const Layout L = layout(P, B, d, 0, Vd, k);
    WF_TRY(check_ws(ws, ws_bytes, L.part));   // control block, keys and top-k candidates
    WF_TRY(check_device());
    WF_TRY(check_local({hidden, W, x, Wd}));
    int num_n2 = 0;
    WF_TRY(launch_lmhead_draft(hidden, W, P, d, V, ids, maxlogit, x, Wd, B, Vd, k, ws, L.cand, lse ? L.lsep : 0,
                               &num_n2, stream));
    return launch_topk_merge(merge_args(B, Vd, num_n2, k, d2t, draft_ids, tids, vals, ws, L.cand, lse, L.lsep), ws,
                             stream);
}

static bool bad_catchup_shape(int B, int N, int din, int H, int G, int D) {
    if (B < 1 || N < B || din < 8 || din % 8 || din > 16384) return true;
    if (G < 1 || H < G || H % G || H / G > 16 || D < 16 || D % 16 || D > 128) return true;
    if ((long)H * D > 16384) return true;
    return catchup_attend_smem(H, G, D) > 200 * 1024;
}

size_t wf_catchup_workspace_bytes(int B, int N, int din, int H, int G, int D) {
    if (bad_catchup_shape(B, N, din, H, G, D)) return 0;
    return catchup_workspace_bytes(B, N, din, H, G, D);
}

static wf_status check_catchup(const wf_catchup_args* a, void* ws, size_t ws_bytes, bool with_final) {
    if (!a) return WF_ERR_INVALID_ARG;
    if (bad_catchup_shape(a->B, a->N, a->din, a->H, a->G, a->D) || a->cap < 1) return WF_ERR_INVALID_ARG;
    if ((long long)a->B * a->cap > 0x7FFFFFFFll - 4096) return WF_ERR_INVALID_ARG;   // cache rows as int coordinates
    if (!a->u || !a->bl_off || !a->cache_len || !a->gamma || !a->Wk || !a->Wv || !a->Kc || !a->Vc)
        return WF_ERR_INVALID_ARG;
    if (with_final && (!a->Wq || !a->Wo || !a->out)) return WF_ERR_INVALID_ARG;
    if (!(a->eps >= 0.f) || !(a->theta > 0.f)) return WF_ERR_INVALID_ARG;
    if (!aligned16(a->u) || !aligned16(a->gamma) || !aligned16(a->Wk) || !aligned16(a->Wv) || !aligned16(a->Kc) ||
        !aligned16(a->Vc))
        return WF_ERR_INVALID_ARG;
    if (with_final && (!aligned16(a->Wq) || !aligned16(a->Wo))) return WF_ERR_INVALID_ARG;
    WF_TRY(check_ws(ws, ws_bytes, catchup_workspace_bytes(a->B, a->N, a->din, a->H, a->G, a->D)));
    WF_TRY(check_device());
    // the projections read the weights and the normalised rows (in the workspace) by TMA
    return check_local({a->u, a->Wk, a->Wv, a->Wq, a->Wo, a->Kc, a->Vc, ws});
}

wf_status wf_catchup_kv(const wf_catchup_args* a, void* ws, size_t ws_bytes, wf_stream_t stream) {
    WF_TRY(check_catchup(a, ws, ws_bytes, false));
    return launch_catchup(a, ws, false, stream);
}

wf_status wf_catchup(const wf_catchup_args* a, void* ws, size_t ws_bytes, wf_stream_t stream) {
    WF_TRY(check_catchup(a, ws, ws_bytes, true));
    return launch_catchup(a, ws, true, stream);
}

wf_status wf_round(const wf_round_args* a, void* ws, size_t ws_bytes, wf_stream_t stream) {
    if (!a) return WF_ERR_INVALID_ARG;
    if (!a->hidden || !a->W || bad_gemm_shape(a->P, a->d, a->V)) return WF_ERR_INVALID_ARG;
    if (a->B < 1 || !a->pos_off || !a->node_off || !a->tok) return WF_ERR_INVALID_ARG;
    if (!a->kind && !a->parent) return WF_ERR_INVALID_ARG;
    if (a->path_stride < 0 || (a->path_stride > 0 && !a->path)) return WF_ERR_INVALID_ARG;
    const bool entropy = a->router_kind == WF_ROUTER_ENTROPY;
    if (a->router_kind != WF_ROUTER_NEURAL && !entropy) return WF_ERR_INVALID_ARG;
    if (!entropy && (a->m < 1 || a->m > ROUTER_MAX_WIDTH || !a->W1 || !a->b1 || !a->w2)) return WF_ERR_INVALID_ARG;
    if (entropy && a->P > ROUTE_ALL_ROWS_MAX && a->B > ENT_MAX_ROWS) return WF_ERR_UNSUPPORTED;
    if (!a->ids || !a->n_accept || !a->bonus || !a->last_pos || !a->delta_al || !a->route) return WF_ERR_INVALID_ARG;
    if (!aligned16(a->hidden) || !aligned16(a->W) || (!entropy && !aligned16(a->W1))) return WF_ERR_INVALID_ARG;
    const bool draft = a->Wd != nullptr;
    if (draft) {
        if (!a->x || !a->d2t || !a->tids || bad_gemm_shape(a->B, a->d, a->Vd)) return WF_ERR_INVALID_ARG;
        if (a->k < 1 || a->k > WF_MAX_TOPK || a->k > a->Vd) return WF_ERR_INVALID_ARG;
        if (!aligned16(a->x) || !aligned16(a->Wd)) return WF_ERR_INVALID_ARG;
    }
    const Layout L = layout(a->P, a->B, a->d, entropy ? 1 : a->m, draft ? a->Vd : 0, draft ? a->k : 0);
    WF_TRY(check_ws(ws, ws_bytes, L.total));
    WF_TRY(check_device());
    WF_TRY(check_local({a->hidden, a->W, draft ? a->x : nullptr, draft ? a->Wd : nullptr, entropy ? ws : nullptr}));
    float* dall = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + L.dall);
    if (entropy && a->P <= ROUTE_ALL_ROWS_MAX) {
        // WhiFlash-Entropy, few rows: the LM-head sweep also yields the entropy
        // of every row; acceptance picks the accepted row's.  With one
        // activation tile per head the draft head shares that sweep and its
        // top-k merge runs in the verification launch.
        // The sweep leaves its per-CTA softmax statistics in the workspace and
        // acceptance merges them at each sequence's accepted row only.
        const bool shared = draft && a->P <= BM && a->B <= BM;
        int num_n2 = 0, nslots = 0;
        if (shared)
            WF_TRY(launch_lmhead_draft(a->hidden, a->W, a->P, a->d, a->V, a->ids, a->maxlogit, a->x, a->Wd, a->B,
                                       a->Vd, a->k, ws, L.cand, a->lse ? L.lsep : 0, &num_n2, stream, nullptr, a->tau,
                                       L.ent, &nslots));
        else
            WF_TRY(launch_lmhead_entropy(a->hidden, a->W, a->P, a->d, a->V, a->ids, a->maxlogit, nullptr, nullptr,
                                         a->tau, nullptr, 0, ws, L.ent, stream, &nslots));
        const MergeArgs mg = merge_args(a->B, a->Vd, num_n2, a->k, a->d2t, a->draft_ids, a->tids, a->vals, ws,
                                        L.cand, a->lse, L.lsep);
        const float4* ent = reinterpret_cast<const float4*>(reinterpret_cast<const uint8_t*>(ws) + L.ent);
        WF_TRY(launch_verify(a->ids, a->tok, a->parent, a->kind, 1, a->pos_off, a->node_off, a->B, a->P,
                             a->path ? a->path_stride : 0, a->n_accept, a->bonus, a->last_pos, a->path, ws, stream,
                             RoutePick{nullptr, ent, nslots, a->tau, a->delta_al, a->route}, true,
                             shared ? &mg : nullptr));
        if (shared) return WF_OK;
    } else if (entropy) {
        // many rows: a second sweep over the weights for the B accepted rows
        // only.  The draft head rides in the first sweep (paired CTAs) when its
        // rows fit one tile pair; its merge then runs beside the verification.
        const bool shared = draft && a->B <= 2 * BM;
        int num_n2 = 0;
        if (shared)
            WF_TRY(launch_lmhead_draft(a->hidden, a->W, a->P, a->d, a->V, a->ids, a->maxlogit, a->x, a->Wd, a->B,
                                       a->Vd, a->k, ws, L.cand, a->lse ? L.lsep : 0, &num_n2, stream));
        else
            WF_TRY(launch_lmhead_argmax(a->hidden, a->W, a->P, a->d, a->V, a->ids, a->maxlogit, ws, stream));
        const MergeArgs mg = merge_args(a->B, a->Vd, num_n2, a->k, a->d2t, a->draft_ids, a->tids, a->vals, ws,
                                        L.cand, a->lse, L.lsep);
        WF_TRY(launch_verify(a->ids, a->tok, a->parent, a->kind, 1, a->pos_off, a->node_off, a->B, a->P,
                             a->path ? a->path_stride : 0, a->n_accept, a->bonus, a->last_pos, a->path, ws, stream,
                             RoutePick{}, true, shared ? &mg : nullptr));
        uint16_t* gath = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(ws) + L.gath);
        WF_TRY(launch_gather_rows(a->hidden, a->P, a->d, a->last_pos, a->B, gath, ws, stream));
        WF_TRY(launch_lmhead_entropy(gath, a->W, a->B, a->d, a->V, nullptr, nullptr, a->delta_al, a->route, a->tau,
                                     a->last_pos, a->P, ws, L.ent, stream));
        if (shared) return WF_OK;
    } else {
        // Neural router.  With few rows it runs on every verified row beside
        // the LM head (it needs only the hidden states and its weights, and
        // waits for the LM head just before it exits) and acceptance picks the
        // accepted row's output; otherwise it routes each sequence's accepted
        // row after acceptance, its weights already loaded while acceptance
        // runs.  The draft head shares the LM head's weight sweep (its tiles
        // first) when each head fits one activation tile, or, with several
        // activation tiles, when the draft rows fit one tile pair of the paired
        // sweep; its candidates are merged beside the verification.
        const bool beside = a->P <= ROUTER_BESIDE_MAX_ROWS;
        const bool shared = draft && (a->P <= BM ? a->B <= BM : a->B <= 2 * BM);
        int num_n2 = 0;
        if (shared)
            WF_TRY(launch_lmhead_draft(a->hidden, a->W, a->P, a->d, a->V, a->ids, a->maxlogit, a->x, a->Wd, a->B,
                                       a->Vd, a->k, ws, L.cand, a->lse ? L.lsep : 0, &num_n2, stream));
        else
            WF_TRY(launch_lmhead_argmax(a->hidden, a->W, a->P, a->d, a->V, a->ids, a->maxlogit, ws, stream));
        // the shared sweep's candidate lists are merged by extra CTAs of the
        // verification launch, beside the verification
        const MergeArgs mg = merge_args(a->B, a->Vd, num_n2, a->k, a->d2t, a->draft_ids, a->tids, a->vals, ws,
                                        L.cand, a->lse, L.lsep);
        const MergeArgs* mgp = shared ? &mg : nullptr;
        if (beside) {
            WF_TRY(launch_router(a->hidden, nullptr, a->P, a->d, a->m, a->P, a->W1, a->b1, a->w2, a->b2, a->tau, dall,
                                 nullptr, ws, L.part, stream));
            WF_TRY(launch_verify(a->ids, a->tok, a->parent, a->kind, 1, a->pos_off, a->node_off, a->B, a->P,
                                 a->path ? a->path_stride : 0, a->n_accept, a->bonus, a->last_pos, a->path, ws,
                                 stream, RoutePick{dall, nullptr, 0, a->tau, a->delta_al, a->route}, true, mgp));
        } else {
            WF_TRY(launch_verify(a->ids, a->tok, a->parent, a->kind, 1, a->pos_off, a->node_off, a->B, a->P,
                                 a->path ? a->path_stride : 0, a->n_accept, a->bonus, a->last_pos, a->path, ws,
                                 stream, RoutePick{}, true, mgp));
            WF_TRY(launch_router(a->hidden, a->last_pos, a->B, a->d, a->m, a->P, a->W1, a->b1, a->w2, a->b2, a->tau,
                                 a->delta_al, a->route, ws, L.part, stream));
        }
        if (shared) return WF_OK;
        if (draft)
            WF_TRY(launch_draft_topk(a->x, a->Wd, a->d2t, a->B, a->d, a->Vd, a->k, a->draft_ids, a->tids, a->vals,
                                     a->lse, ws, L.cand, L.lsep, stream));
        return WF_OK;
    }
    if (draft)
        WF_TRY(launch_draft_topk(a->x, a->Wd, a->d2t, a->B, a->d, a->Vd, a->k, a->draft_ids, a->tids, a->vals,
                                 a->lse, ws, L.cand, L.lsep, stream));
    return WF_OK;
}

}  // extern "C"
