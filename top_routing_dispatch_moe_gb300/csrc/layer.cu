// The layer forward as one C call: router -> dispatch -> grouped SwiGLU experts -> combine ("Megatron-LM
// 分布式训练（六）", section "MoE 层的数据流"; "v6 长序列和 MoE", the worked shape table), with token-choice,
// Sinkhorn-balanced or expert-choice routing ("10.5 序列并行与专家并行", section 10.5.6) and the bf16 / fp32 or the
// FP8 send buffer (section 10.5.7), and the same over batches in page-locked host memory with the host <-> device
// copies overlapped with the layer.
//
// Host code only: every step is one of the library's own entry points, enqueued on the caller's stream over
// intermediates laid out in one caller-provided workspace. Each step, and each batch of the host variant, is an NVTX
// range ("moe.router", "moe.dispatch", "moe.up_gate", "moe.down", "moe.shared", "moe.combine", "moe.batch"), so that
// a profiler can attribute the launches (e.g. ncu --nvtx --nvtx-include "moe.up_gate/"); without a profiler attached
// the ranges cost a branch each. Nothing here allocates device memory; the host variant
// creates two copy streams and a few events per call and releases them before it returns (the runtime frees them
// once the work they order has completed).
#include <stdio.h>
#include <vector>
#include <nvtx3/nvToolsExt.h>
#include "common.cuh"

namespace moe {
namespace {

// Byte offsets of the intermediates inside the workspace, each region 256-byte aligned.
struct LayerLayout {
    size_t logits, ids, gates, counts, f, P, aux, router_ws, router_ws_bytes;
    size_t buf, offsets, kept, dest_row, drop_mask, src_token, src_slot, rank_counts, rank_offsets, sched;
    size_t disp_ws, disp_ws_bytes;
    size_t ec_tokens, ec_gates, ec_slot, ec_ws, ec_ws_bytes;        // expert choice
    size_t sel_bias, sk_ws, sk_ws_bytes, rl_ws, rl_ws_bytes;          // Sinkhorn
    size_t buf8, scales;                                              // FP8 payload
    size_t act, eout, sh_sched, sh_act, sh_out;
    size_t fwd_bytes;        // end of the forward's regions
    size_t x_dev[2], y_dev[2];
    size_t host_bytes;       // end of the host variant's regions
    long long rows;
};

size_t el_size(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }

LayerLayout layout_of(const moe_layer_desc& d) {
    LayerLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    const size_t T = (size_t)d.T, h = (size_t)d.h, E = (size_t)d.E, k = (size_t)d.k, F = (size_t)d.F;
    const size_t el = el_size(d.dtype);
    const bool ec = d.routing == MOE_ROUTING_EXPERT_CHOICE;
    L.rows = ec ? (long long)d.E * d.capacity : (long long)moe_dispatch_rows(d.T, d.E, d.k, d.capacity);
    const size_t rows = (size_t)L.rows;
    L.logits = take(T * E * 4);
    L.ids = take(T * k * 4);
    L.gates = take(T * k * 4);
    L.counts = take(E * 4);
    L.f = take(E * 4);
    L.P = take(E * 4);
    L.aux = take(4);
    L.router_ws_bytes = moe_router_workspace_size(d.T, d.h, d.E, d.k, d.dtype);
    L.router_ws = take(L.router_ws_bytes);
    L.buf = take(rows * h * el);
    if (ec) {
        L.ec_tokens = take(E * (size_t)d.capacity * 4);
        L.ec_gates = take(E * (size_t)d.capacity * 4);
        L.ec_slot = take(T * E * 4);
        L.ec_ws_bytes = moe_expert_choice_workspace_size(d.T, d.E);
        L.ec_ws = take(L.ec_ws_bytes);
        L.sched = take(moe_tile_sched_bytes(d.T, d.E, 1, d.capacity));
    } else {
        L.offsets = take((E + 1) * 4);
        L.kept = take(E * 4);
        L.dest_row = take(T * k * 4);
        L.drop_mask = take(T * k);
        L.src_token = take(rows * 4);
        L.src_slot = take(rows * 4);
        L.rank_counts = take((size_t)d.num_ranks * 4);
        L.rank_offsets = take(((size_t)d.num_ranks + 1) * 4);
        L.sched = take(moe_tile_sched_bytes(d.T, d.E, d.k, d.capacity));
        L.disp_ws_bytes = moe_dispatch_workspace_size(d.T, d.E, d.k, d.capacity);
        L.disp_ws = take(L.disp_ws_bytes);
    }
    if (d.routing == MOE_ROUTING_SINKHORN) {
        L.sel_bias = take(E * 4);
        L.sk_ws_bytes = moe_sinkhorn_workspace_size(d.T, d.E);
        L.sk_ws = take(L.sk_ws_bytes);
        L.rl_ws_bytes = moe_router_from_logits_workspace_size(d.T, d.E);
        L.rl_ws = take(L.rl_ws_bytes);
    }
    if (d.payload == MOE_PAYLOAD_FP8) {       // the e4m3 send buffer; buf receives its dequantised rows
        L.buf8 = take(rows * h);
        L.scales = take(rows * (h / 128) * 4);
    }
    L.act = take(rows * F * el);
    L.eout = take(rows * h * el);
    if (d.packed_shared) {
        L.sh_sched = take(moe_tile_sched_bytes(d.T, 1, 1, 0));
        L.sh_act = take(T * F * el);
        L.sh_out = take(T * h * el);
    }
    L.fwd_bytes = o;
    for (int b = 0; b < 2; ++b) L.x_dev[b] = take(T * h * el);
    for (int b = 0; b < 2; ++b) L.y_dev[b] = take(T * h * el);
    L.host_bytes = o;
    return L;
}

int check_desc(const moe_layer_desc* d, const char* who) {
    MOE_REQUIRE(d, MOE_ERR_INVALID_ARG, "%s: desc is NULL", who);
    MOE_REQUIRE(d->dtype == MOE_BF16 || d->dtype == MOE_F32, MOE_ERR_UNSUPPORTED, "%s: dtype %d", who, d->dtype);
    MOE_REQUIRE(d->routing == MOE_ROUTING_TOKEN || d->routing == MOE_ROUTING_EXPERT_CHOICE ||
                    d->routing == MOE_ROUTING_SINKHORN,
                MOE_ERR_UNSUPPORTED, "%s: routing %d", who, d->routing);
    MOE_REQUIRE(d->payload == MOE_PAYLOAD_DTYPE || d->payload == MOE_PAYLOAD_FP8, MOE_ERR_UNSUPPORTED, "%s: payload %d",
                who, d->payload);
    MOE_REQUIRE(d->routing == MOE_ROUTING_SINKHORN || d->gating == MOE_GATING_SOFTMAX ||
                    d->gating == MOE_GATING_SOFTMAX_RENORM || d->gating == MOE_GATING_SIGMOID_BIAS_RENORM,
                MOE_ERR_UNSUPPORTED, "%s: gating %d (the selection-bias mode is Sinkhorn routing's)", who, d->gating);
    MOE_REQUIRE(d->payload != MOE_PAYLOAD_FP8 || (d->dtype == MOE_BF16 && d->routing == MOE_ROUTING_TOKEN),
                MOE_ERR_UNSUPPORTED, "%s: the FP8 payload needs bf16 and token-choice routing", who);
    MOE_REQUIRE(d->payload != MOE_PAYLOAD_FP8 || d->h % 128 == 0, MOE_ERR_INVALID_ARG,
                "%s: the FP8 payload needs h %% 128 == 0 (h=%d)", who, d->h);
    MOE_REQUIRE(d->routing != MOE_ROUTING_EXPERT_CHOICE || (d->capacity >= 1 && d->capacity <= d->T && d->E <= 256),
                MOE_ERR_INVALID_ARG, "%s: expert choice needs 1 <= capacity <= T and E <= 256 (C=%d T=%d E=%d)", who,
                d->capacity, d->T, d->E);
    MOE_REQUIRE(d->sinkhorn_iters >= 0, MOE_ERR_INVALID_ARG, "%s: sinkhorn_iters %d", who, d->sinkhorn_iters);
    MOE_REQUIRE(d->T >= 0 && d->h > 0 && d->h % 8 == 0 && d->F > 0 && d->F % 8 == 0 && d->E >= 1 && d->E <= 1024 &&
                    d->k >= 1 && d->k <= 16 && d->k <= d->E && d->capacity >= 0 && d->num_ranks >= 1 &&
                    d->E % d->num_ranks == 0,
                MOE_ERR_INVALID_ARG, "%s: T=%d h=%d E=%d k=%d F=%d capacity=%d num_ranks=%d", who, d->T, d->h, d->E,
                d->k, d->F, d->capacity, d->num_ranks);
    MOE_REQUIRE(d->w_r_packed && aligned16(d->w_r_packed) && d->packed_w && aligned16(d->packed_w) &&
                    (!d->packed_shared || aligned16(d->packed_shared)) && (!d->bias || aligned16(d->bias)),
                MOE_ERR_INVALID_ARG, "%s: w_r_packed and packed_w must be non-null, all parameters 16-byte aligned",
                who);
    return MOE_OK;
}

template <class T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// One NVTX range for the lifetime of the object (the enqueueing of one step on the host).
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
};

moe_layer_views views_at(const moe_layer_desc& d, const LayerLayout& L, void* ws) {
    moe_layer_views v{};
    v.logits = at<float>(ws, L.logits);
    v.topk_ids = at<int32_t>(ws, L.ids);
    v.gates = at<float>(ws, L.gates);
    v.counts = at<int32_t>(ws, L.counts);
    v.f = at<float>(ws, L.f);
    v.P = at<float>(ws, L.P);
    v.aux = at<float>(ws, L.aux);
    v.buf = at<void>(ws, L.buf);
    v.tile_sched = at<int32_t>(ws, L.sched);
    if (d.routing == MOE_ROUTING_EXPERT_CHOICE) {
        v.ec_tokens = at<int32_t>(ws, L.ec_tokens);
        v.ec_gates = at<float>(ws, L.ec_gates);
        v.ec_slot = at<int32_t>(ws, L.ec_slot);
    } else {
        v.offsets = at<int32_t>(ws, L.offsets);
        v.kept_counts = at<int32_t>(ws, L.kept);
        v.dest_row = at<int32_t>(ws, L.dest_row);
        v.drop_mask = at<uint8_t>(ws, L.drop_mask);
        v.src_token = at<int32_t>(ws, L.src_token);
        v.src_slot = at<int32_t>(ws, L.src_slot);
        v.rank_counts = at<int32_t>(ws, L.rank_counts);
        v.rank_offsets = at<int32_t>(ws, L.rank_offsets);
    }
    if (d.routing == MOE_ROUTING_SINKHORN) v.sel_bias = at<float>(ws, L.sel_bias);
    if (d.payload == MOE_PAYLOAD_FP8) {
        v.buf8 = at<uint8_t>(ws, L.buf8);
        v.scales = at<float>(ws, L.scales);
    }
    v.act = at<void>(ws, L.act);
    v.eout = at<void>(ws, L.eout);
    v.act_shared = d.packed_shared ? at<void>(ws, L.sh_act) : nullptr;
    v.out_shared = d.packed_shared ? at<void>(ws, L.sh_out) : nullptr;
    v.rows = L.rows;
    return v;
}

// The chain on one stream. With bf16 and the dtype payload a shared expert runs its tiles inside the routed
// launches (as moe_expert_up_gate_shared / moe_expert_down_shared); otherwise it runs as a dense group of its own.
int forward_chain(const moe_layer_desc& d, const LayerLayout& L, const void* x, void* y, void* ws, void* s) {
    const moe_layer_views v = views_at(d, L, ws);
    const int rows = (int)L.rows;
    const bool ec = d.routing == MOE_ROUTING_EXPERT_CHOICE, sk = d.routing == MOE_ROUTING_SINKHORN;
    const bool fused_shared = d.packed_shared && d.dtype == MOE_BF16 && d.payload == MOE_PAYLOAD_DTYPE;
    int rc;
    {
        Range r("moe.router");
        rc = moe_router_packed(x, d.w_r_packed, d.bias, d.T, d.h, d.E, d.k, d.dtype, sk ? MOE_GATING_SOFTMAX : d.gating,
                               d.alpha, v.logits, v.topk_ids, v.gates, v.counts, v.f, v.P, v.aux,
                               at<void>(ws, L.router_ws), L.router_ws_bytes, s);
        if (rc) return rc;
        if (sk) {                            // balanced selection: the Sinkhorn log column scalings as a bias
            rc = moe_sinkhorn_bias(v.logits, d.T, d.E, d.sinkhorn_iters > 0 ? d.sinkhorn_iters : 16, v.sel_bias,
                                   at<void>(ws, L.sk_ws), L.sk_ws_bytes, s);
            if (rc) return rc;
            rc = moe_router_from_logits(v.logits, v.sel_bias, d.T, d.E, d.k, MOE_GATING_SOFTMAX_SELBIAS, d.alpha,
                                        v.topk_ids, v.gates, v.counts, v.f, v.P, v.aux, at<void>(ws, L.rl_ws),
                                        L.rl_ws_bytes, s);
            if (rc) return rc;
        }
        if (ec) {
            rc = moe_expert_choice_route(v.logits, d.T, d.E, d.capacity, v.ec_tokens, v.ec_gates, v.ec_slot,
                                         at<void>(ws, L.ec_ws), L.ec_ws_bytes, s);
            if (rc) return rc;
        }
    }
    {
        Range r("moe.dispatch");
        if (ec) {
            rc = moe_expert_choice_dispatch(x, v.ec_tokens, d.T, d.h, d.E, d.capacity, d.dtype, v.buf, v.tile_sched,
                                            s);
        } else if (d.payload == MOE_PAYLOAD_FP8) {
            rc = moe_dispatch_fp8(x, v.topk_ids, d.T, d.h, d.E, d.k, d.capacity, d.num_ranks, v.buf8, v.scales,
                                  v.offsets, v.kept_counts, v.dest_row, v.drop_mask, v.src_token, v.src_slot,
                                  v.rank_counts, v.rank_offsets, v.tile_sched, at<void>(ws, L.disp_ws),
                                  L.disp_ws_bytes, s);
            if (!rc) rc = moe_dequant_fp8(v.buf8, v.scales, rows, d.h, v.buf, s);   // receive side, then bf16 GEMMs
        } else {
            rc = moe_dispatch(x, v.topk_ids, d.T, d.h, d.E, d.k, d.capacity, d.num_ranks, d.dtype, v.buf, v.offsets,
                              v.kept_counts, v.dest_row, v.drop_mask, v.src_token, v.src_slot, v.rank_counts,
                              v.rank_offsets, v.tile_sched, at<void>(ws, L.disp_ws), L.disp_ws_bytes, s);
        }
        if (rc) return rc;
    }
    {
        Range r("moe.up_gate");
        rc = fused_shared ? moe_expert_up_gate_shared(v.buf, v.tile_sched, d.packed_w, d.E, d.h, d.F, rows, x, d.T,
                                                      d.packed_shared, v.act_shared, d.dtype, v.act, s)
                          : moe_expert_up_gate(v.buf, v.tile_sched, d.packed_w, d.E, d.h, d.F, rows, d.dtype, v.act, s);
        if (rc) return rc;
    }
    {
        Range r("moe.down");
        rc = fused_shared ? moe_expert_down_shared(v.act, v.tile_sched, d.packed_w, d.E, d.h, d.F, rows, v.act_shared,
                                                   d.T, d.packed_shared, v.out_shared, d.dtype, v.eout, s)
                          : moe_expert_down(v.act, v.tile_sched, d.packed_w, d.E, d.h, d.F, rows, d.dtype, v.eout, s);
        if (rc) return rc;
    }
    if (d.packed_shared && !fused_shared) {  // the shared expert as a dense group of T rows
        Range r("moe.shared");
        int32_t* sh_sched = at<int32_t>(ws, L.sh_sched);
        rc = moe_dense_tile_sched(d.T, sh_sched, s);
        if (!rc) rc = moe_expert_up_gate(x, sh_sched, d.packed_shared, 1, d.h, d.F, d.T, d.dtype, v.act_shared, s);
        if (!rc) rc = moe_expert_down(v.act_shared, sh_sched, d.packed_shared, 1, d.h, d.F, d.T, d.dtype, v.out_shared, s);
        if (rc) return rc;
    }
    Range r("moe.combine");
    if (ec)
        return moe_expert_choice_combine(v.eout, v.ec_slot, v.ec_gates, v.out_shared, d.T, d.h, d.E, d.capacity,
                                         d.dtype, y, s);
    return moe_combine(v.eout, v.dest_row, v.gates, v.out_shared, d.T, d.h, d.k, d.dtype, y, s);
}

bool page_locked(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();                  // clear the sticky-free error of an unknown pointer
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// Releases the copy streams and events of one host-variant call (deferred by the runtime until their work ends).
struct HostCallObjects {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    std::vector<cudaEvent_t> events;
    ~HostCallObjects() {
        for (cudaEvent_t e : events) cudaEventDestroy(e);
        if (h2d) cudaStreamDestroy(h2d);
        if (d2h) cudaStreamDestroy(d2h);
    }
    cudaEvent_t event() {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        events.push_back(e);
        return e;
    }
};

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_layer_workspace_size(const moe_layer_desc* desc) {
    return desc ? layout_of(*desc).fwd_bytes : 0;
}

extern "C" size_t moe_layer_host_workspace_size(const moe_layer_desc* desc) {
    return desc ? layout_of(*desc).host_bytes : 0;
}

extern "C" int moe_layer_views_of(const moe_layer_desc* desc, void* ws, moe_layer_views* views) {
    if (int rc = check_desc(desc, "moe_layer_views_of")) return rc;
    MOE_REQUIRE(ws && aligned16(ws) && views, MOE_ERR_INVALID_ARG, "moe_layer_views_of: null or misaligned ws / views");
    *views = views_at(*desc, layout_of(*desc), ws);
    return MOE_OK;
}

extern "C" int moe_layer_forward(const moe_layer_desc* desc, const void* x, void* y, void* ws, size_t ws_bytes,
                                 void* stream) {
    if (int rc = check_desc(desc, "moe_layer_forward")) return rc;
    const LayerLayout L = layout_of(*desc);
    MOE_REQUIRE(x && y && ws && aligned16(x) && aligned16(y) && aligned16(ws), MOE_ERR_INVALID_ARG,
                "moe_layer_forward: x, y and ws must be non-null and 16-byte aligned");
    MOE_REQUIRE(ws_bytes >= L.fwd_bytes, MOE_ERR_WORKSPACE, "moe_layer_forward: workspace %zu < %zu bytes", ws_bytes,
                L.fwd_bytes);
    if (desc->T == 0) return MOE_OK;
    return forward_chain(*desc, L, x, y, ws, stream);
}

extern "C" int moe_layer_forward_host(const moe_layer_desc* desc, int n_batches, const void* const* x_host,
                                      void* const* y_host, void* ws, size_t ws_bytes, void* stream) {
    if (int rc = check_desc(desc, "moe_layer_forward_host")) return rc;
    const LayerLayout L = layout_of(*desc);
    MOE_REQUIRE(n_batches >= 0 && (n_batches == 0 || (x_host && y_host)) && ws && aligned16(ws), MOE_ERR_INVALID_ARG,
                "moe_layer_forward_host: n_batches=%d, x_host / y_host / ws null or ws misaligned", n_batches);
    MOE_REQUIRE(ws_bytes >= L.host_bytes, MOE_ERR_WORKSPACE, "moe_layer_forward_host: workspace %zu < %zu bytes",
                ws_bytes, L.host_bytes);
    for (int i = 0; i < n_batches; ++i)
        MOE_REQUIRE(x_host[i] && y_host[i] && page_locked(x_host[i]) && page_locked(y_host[i]), MOE_ERR_INVALID_ARG,
                    "moe_layer_forward_host: batch %d: x_host and y_host must be page-locked host memory", i);
    if (n_batches == 0 || desc->T == 0) return MOE_OK;
    const size_t bytes = (size_t)desc->T * desc->h * el_size(desc->dtype);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    HostCallObjects o;
    cudaError_t e = cudaStreamCreateWithFlags(&o.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&o.d2h, cudaStreamNonBlocking);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "moe_layer_forward_host: stream: %s", cudaGetErrorString(e));
    // the first copies start after the work already enqueued on `stream` (which may still use the buffers)
    cudaEvent_t start = o.event();
    MOE_REQUIRE(start, MOE_ERR_CUDA, "moe_layer_forward_host: event creation failed");
    e = cudaEventRecord(start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(o.h2d, start, 0);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "moe_layer_forward_host: start: %s", cudaGetErrorString(e));
    cudaEvent_t x_free[2] = {nullptr, nullptr};    // the layer has finished reading x buffer b
    cudaEvent_t y_free[2] = {nullptr, nullptr};    // the copy out of y buffer b has finished
    cudaEvent_t last_in = nullptr;                 // the last copy in that was issued
    // `stream` waits for every copy issued so far, on success and on every error path alike, so that a caller who
    // synchronises `stream` may then reuse or free the host buffers
    auto join = [&]() {
        cudaError_t j = cudaSuccess;
        for (cudaEvent_t ev : {last_in, y_free[0], y_free[1]})
            if (ev && j == cudaSuccess) j = cudaStreamWaitEvent(s, ev, 0);
        return j;
    };
    auto fail = [&](int code, int batch, const char* step, cudaError_t err) {
        join();
        char inner[512];                     // the failing call's own message (set_error rewrites that buffer)
        snprintf(inner, sizeof(inner), "%s", err == cudaSuccess ? moe_last_error_string() : cudaGetErrorString(err));
        return set_error(code, "moe_layer_forward_host: batch %d %s: %s", batch, step, inner);
    };
    for (int i = 0; i < n_batches; ++i) {
        const int b = i & 1;
        void* xd = at<void>(ws, L.x_dev[b]);
        void* yd = at<void>(ws, L.y_dev[b]);
        cudaEvent_t x_in = o.event(), done = o.event(), out = o.event();
        if (!x_in || !done || !out) return fail(MOE_ERR_CUDA, i, "event creation", cudaErrorMemoryAllocation);
        if (x_free[b]) e = cudaStreamWaitEvent(o.h2d, x_free[b], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(xd, x_host[i], bytes, cudaMemcpyHostToDevice, o.h2d);
        if (e == cudaSuccess) e = cudaEventRecord(x_in, o.h2d);
        if (e == cudaSuccess) last_in = x_in;
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, x_in, 0);
        if (e == cudaSuccess && y_free[b]) e = cudaStreamWaitEvent(s, y_free[b], 0);
        if (e != cudaSuccess) return fail(MOE_ERR_CUDA, i, "copy in", e);
        {
            Range r("moe.batch");
            if (int rc = forward_chain(*desc, L, xd, yd, ws, stream)) return fail(rc, i, "layer", cudaSuccess);
        }
        e = cudaEventRecord(done, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(o.d2h, done, 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(y_host[i], yd, bytes, cudaMemcpyDeviceToHost, o.d2h);
        if (e == cudaSuccess) e = cudaEventRecord(out, o.d2h);
        if (e != cudaSuccess) return fail(MOE_ERR_CUDA, i, "copy out", e);
        x_free[b] = done;
        y_free[b] = out;
    }
    if ((e = join()) != cudaSuccess)
        return set_error(MOE_ERR_CUDA, "moe_layer_forward_host: join: %s", cudaGetErrorString(e));
    return MOE_OK;
}
