// C ABI entry points: argument checks, workspace carving and the ordered
// launch sequence of the layer.  No entry point allocates, frees or
// synchronises (mok_get_error excepted, see status.cu).
#include "common.cuh"
#include "kernels.h"

namespace mok {

bool shape_ok(const mok_shape* s) {
  if (!s) return false;
  if (s->T < 0 || s->D <= 0 || s->I <= 0 || s->E < 1 || s->E > 1024 || s->K < 1 || s->K > 32 ||
      s->K > s->E || s->I_shared < 0)
    return false;
  if (s->D % 256 || s->I % 128 || s->I_shared % 128) return false;
  if (static_cast<int64_t>(s->T) * s->K >= (int64_t(1) << 31)) return false;
  if (s->dtype != MOK_BF16 && s->dtype != MOK_MXFP8) return false;
  if (s->chunk_rows != 0 && s->chunk_rows != -1 && (s->chunk_rows < 512 || s->chunk_rows > 32768)) return false;
  if (s->producer_sms < 0 || s->producer_sms > 4096) return false;
  if (s->bwd_shared_sms < 0 || s->bwd_shared_sms > 4096) return false;
  return true;
}

int shared_expert_sms(const mok_shape& s) {
  if (s.producer_sms <= 0) return 0;
  const int left = num_sms() - s.producer_sms;
  return left >= 2 ? left : 2;
}

int bwd_shared_split(const mok_shape& s) {
  if (!s.I_shared || s.bwd_shared_sms <= 0 || s.T == 0) return 0;
  const int cap = num_sms() / 3;
  const int k = s.bwd_shared_sms < cap ? s.bwd_shared_sms : cap;
  return k >= 2 ? k : 0;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Workspace carving: a bump allocator over the caller's buffer.
struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += round_up(bytes);
    return o;
  }
};

struct FwdLayout {
  size_t topk, g, counts, offsets, table, route_dst, hist, xg, xg_scale, a, a_scale, yg, as, ys,
      ring_counters, total;
};

// Whether the BF16 forward gathers through the ring (no xg): chunk_rows > 0,
// or 0 (automatic) for layers whose GEMMs run row-major tiles, where the
// ring measured faster than the whole-batch dispatch (the skewed 16384-token
// layer: 3.51 vs 3.61 ms at b = 2048); -1 never.
bool uses_ring(const mok_shape& s) {
  if (s.chunk_rows < 0) return false;
  // MXFP8: the ring of quantised rows when asked for (its automatic choice
  // is the whole-batch quantising dispatch)
  if (s.dtype == MOK_MXFP8) return s.chunk_rows > 0;
  return s.chunk_rows > 0 || !routed_rows_as_n(static_cast<int64_t>(s.T) * s.K, s.E);
}

FwdLayout fwd_layout(const mok_shape& s) {
  const size_t T = s.T, D = s.D, I = s.I, E = s.E, K = s.K, Is = s.I_shared, R = T * K;
  Carve c;
  FwdLayout L;
  L.topk = c.take(R * 4);
  L.g = c.take(R * 4);
  L.counts = c.take(E * 4);
  L.offsets = c.take((E + 1) * 4);
  L.table = c.take(R * 12);
  L.route_dst = c.take(R * 4);
  L.hist = c.take(plan_scratch_bytes(static_cast<int64_t>(R), s.E));
  const bool ring = uses_ring(s);
  const int64_t b = ring_chunk(s.chunk_rows);
  // xg holds the ring when the forward gathers through one
  const int elem = s.dtype == MOK_MXFP8 ? 1 : 2;
  L.xg = c.take(ring ? ring_bytes(static_cast<int64_t>(R), D, b, elem) : R * D * elem);
  L.ring_counters = c.take(ring ? ring_counter_bytes(static_cast<int64_t>(R), b) : 0);
  const bool mx = s.dtype == MOK_MXFP8;
  L.xg_scale = c.take(mx ? mx_scale_bytes(static_cast<int64_t>(R), D, s.E) : 0);
  L.a = c.take(R * I * 2);
  L.a_scale = c.take(mx ? mx_scale_bytes(static_cast<int64_t>(R), I, s.E) : 0);
  L.yg = c.take(R * D * 2);
  L.as = c.take(T * Is * 2);
  L.ys = c.take(Is ? T * D * 2 : 0);
  L.total = c.off;
  return L;
}

struct BwdLayout {
  size_t xg, dyg, g_route, dh, du, ag, dgp, dxr, dhs, dus, ags, dxs;
  // MXFP8: x, dY codes and grouped scales; replay h, u and t (bf16); the
  // codes and grouped scales of [dh | du]
  size_t xq, xq_sc, dyq, dyq_sc, hh, uu, tt, dhu_q, dhu_sc;
  size_t total;
};

BwdLayout bwd_layout(const mok_shape& s) {
  const size_t T = s.T, D = s.D, I = s.I, K = s.K, Is = s.I_shared, R = T * K;
  Carve c;
  BwdLayout L;
  L.xg = c.take(R * D * 2);
  L.dyg = c.take(R * D * 2);
  L.g_route = c.take(R * 4);
  L.dh = c.take(R * I * 2);
  L.du = c.take(R * I * 2);
  L.ag = c.take(R * I * 2);
  L.dgp = c.take(R * (I / 32) * 4);
  L.dxr = c.take(R * D * 2);
  L.dhs = c.take(T * Is * 2);
  L.dus = c.take(T * Is * 2);
  L.ags = c.take(T * Is * 2);
  L.dxs = c.take(Is ? T * D * 2 : 0);
  const bool mx = s.dtype == MOK_MXFP8;
  L.xq = c.take(mx ? R * D : 0);
  L.xq_sc = c.take(mx ? mx_scale_bytes(static_cast<int64_t>(R), D, s.E) : 0);
  L.dyq = c.take(mx ? R * D : 0);
  L.dyq_sc = c.take(mx ? mx_scale_bytes(static_cast<int64_t>(R), D, s.E) : 0);
  L.hh = c.take(mx ? R * I * 4 : 0);  // fp32 h, u, t: no rounding point there
  L.uu = c.take(mx ? R * I * 4 : 0);
  L.tt = c.take(mx ? R * I * 4 : 0);
  L.dhu_q = c.take(mx ? R * 2 * I : 0);
  L.dhu_sc = c.take(mx ? mx_scale_bytes(static_cast<int64_t>(R), 2 * I, s.E) : 0);
  L.total = c.off;
  return L;
}

bool mx_bwd_weights_ok(const mok_weights* w) {
  return w->qt_down && w->sct_down && w->qt_gu && w->sct_gu && aligned16(w->qt_down) && aligned16(w->sct_down) &&
         aligned16(w->qt_gu) && aligned16(w->sct_gu);
}

bool mx_weights_ok(const mok_weights* w) {
  return w->q_gate && w->q_up && w->q_down && w->sc_gate && w->sc_up && w->sc_down &&
         aligned16(w->q_gate) && aligned16(w->q_up) && aligned16(w->q_down) &&
         aligned16(w->sc_gate) && aligned16(w->sc_up) && aligned16(w->sc_down) &&
         (!w->sc_gu_pair || aligned16(w->sc_gu_pair));
}

// Workspace of mok_expert_ffn: a (bf16), or a codes + scale words (MXFP8).
size_t ffn_ws_bytes(const mok_shape& s) {
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  if (s.dtype == MOK_MXFP8) return round_up(static_cast<size_t>(R) * s.I) + round_up(mx_scale_bytes(R, s.I, s.E));
  return round_up(static_cast<size_t>(R) * s.I * 2);
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// A non-blocking side stream and two events per device and host thread,
// created on first use and kept for the life of the process: mok_moe_fwd
// runs the shared expert on it, forked from and joined back into the
// caller's stream.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream* side_stream() {
  constexpr int kMaxDevices = 64;
  thread_local SideStream per_device[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = per_device[dev];
  if (!ss.s) {
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess ||
        cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess)
      return nullptr;
  }
  return &ss;
}

}  // namespace
}  // namespace mok

using namespace mok;

extern "C" size_t mok_workspace_bytes(const mok_shape* shape, int op) {
  if (!shape_ok(shape)) return 0;
  const mok_shape& s = *shape;
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  switch (op) {
    case MOK_OP_PLAN: return round_up(plan_scratch_bytes(R, s.E));
    case MOK_OP_EXPERT_FFN: return ffn_ws_bytes(s);
    case MOK_OP_SHARED_FFN: return round_up(static_cast<size_t>(s.T) * (s.I_shared ? s.I_shared : 1) * 2);
    case MOK_OP_FWD: return fwd_layout(s).total;
    case MOK_OP_BWD: return bwd_layout(s).total;
    case MOK_OP_RING: {
      const int64_t b = ring_chunk(s.chunk_rows);
      return round_up(ring_bytes(R, s.D, b)) + round_up(ring_counter_bytes(R, b));
    }
  }
  return 0;
}

extern "C" size_t mok_workspace_offset(const mok_shape* shape, int region) {
  if (!shape_ok(shape)) return static_cast<size_t>(-1);
  const BwdLayout L = bwd_layout(*shape);
  switch (region) {
    case MOK_WS_BWD_DH: return L.dh;
    case MOK_WS_BWD_DU: return L.du;
    case MOK_WS_BWD_AG: return L.ag;
  }
  return static_cast<size_t>(-1);
}

extern "C" mok_status mok_dispatch(const mok_shape* shape, const void* x, const int32_t* table,
                                   const int32_t* route_dst, const int32_t* offsets, void* xg, uint8_t* xg_scale,
                                   void* stream) {
  if (!shape_ok(shape)) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  if (R == 0) return MOK_OK;
  if (!x || !route_dst || !xg || !aligned16(x) || !aligned16(xg)) return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s.dtype == MOK_MXFP8) {
    if (!table || !xg_scale || !offsets) return MOK_ERR_INVALID_ARG;
    return launch_dispatch_mxfp8(x, route_dst, table, offsets, s.T, s.K, s.D, s.E, xg, xg_scale, st);
  }
  return launch_dispatch_bf16(x, route_dst, s.T, s.K, s.D, xg, nullptr, nullptr, st);
}

extern "C" mok_status mok_expert_ffn(const mok_shape* shape, const mok_weights* w, const void* xg,
                                     const uint8_t* xg_scale, const int32_t* offsets, void* a_out,
                                     void* yg, void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(shape) || !w) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  if (R == 0) return MOK_OK;
  if (s.dtype == MOK_MXFP8) {
    if (!xg || !xg_scale || !offsets || !yg || a_out || !mx_weights_ok(w) || !aligned16(xg) ||
        !aligned16(xg_scale) || !aligned16(yg))
      return MOK_ERR_INVALID_ARG;
    if (!ws || ws_bytes < ffn_ws_bytes(s) || (reinterpret_cast<uintptr_t>(ws) & 255u))
      return MOK_ERR_WORKSPACE;
    void* aq = ws;
    void* asc = static_cast<uint8_t*>(ws) + round_up(static_cast<size_t>(R) * s.I);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    mok_status r = launch_upgate_mx(xg, xg_scale, R, w->q_gate, w->sc_gate, w->q_up, w->sc_up,
                                    offsets, s.E, s.D, s.I, aq, asc, st, {}, w->sc_gu_pair);
    if (r != MOK_OK) return r;
    return launch_down_mx(aq, asc, R, w->q_down, w->sc_down, offsets, s.E, s.D, s.I, yg, st);
  }
  if (!xg || !offsets || !yg || !w->w_gate || !w->w_up || !w->w_down) return MOK_ERR_INVALID_ARG;
  if (!aligned16(xg) || !aligned16(yg) || !aligned16(w->w_gate) || !aligned16(w->w_up) ||
      !aligned16(w->w_down) || (a_out && !aligned16(a_out)))
    return MOK_ERR_INVALID_ARG;
  void* a = a_out;
  if (!a) {
    if (!ws || ws_bytes < static_cast<size_t>(R) * s.I * 2) return MOK_ERR_WORKSPACE;
    a = ws;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mok_status r = launch_upgate(xg, R, w->w_gate, w->w_up, offsets, s.E, R, s.D, s.I, a, st);
  if (r != MOK_OK) return r;
  return launch_down(a, R, w->w_down, offsets, s.E, R, s.D, s.I, yg, st);
}

extern "C" mok_status mok_expert_upgate(const mok_shape* shape, const mok_weights* w,
                                        const void* xg, const uint8_t* xg_scale,
                                        const int32_t* offsets, void* a, uint8_t* a_scale,
                                        const void* x_shared, void* a_shared, void* stream) {
  if (!shape_ok(shape) || !w) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  if (R == 0) return MOK_OK;
  const bool with_shared = s.I_shared > 0 && x_shared && a_shared;
  if (with_shared && (!w->ws_gate || !w->ws_up || !aligned16(x_shared) || !aligned16(a_shared)))
    return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!xg && !offsets && !a) {  // the shared expert's up/gate alone (a side stream's work)
    if (!with_shared) return MOK_ERR_INVALID_ARG;
    return launch_upgate(x_shared, s.T, w->ws_gate, w->ws_up, nullptr, 1, s.T, s.D, s.I_shared, a_shared, st,
                         shared_expert_sms(s));
  }
  if (s.dtype == MOK_MXFP8) {
    if (!xg || !xg_scale || !offsets || !a || !a_scale || !mx_weights_ok(w) || !aligned16(xg) ||
        !aligned16(xg_scale) || !aligned16(a) || !aligned16(a_scale))
      return MOK_ERR_INVALID_ARG;
    mok_status r = launch_upgate_mx(xg, xg_scale, R, w->q_gate, w->sc_gate, w->q_up, w->sc_up, offsets,
                                    s.E, s.D, s.I, a, a_scale, st, {}, w->sc_gu_pair);
    if (r != MOK_OK || !with_shared) return r;
    return launch_upgate(x_shared, s.T, w->ws_gate, w->ws_up, nullptr, 1, s.T, s.D, s.I_shared,
                         a_shared, st);
  }
  if (!xg || !offsets || !a || !w->w_gate || !w->w_up || !aligned16(xg) || !aligned16(a) ||
      !aligned16(w->w_gate) || !aligned16(w->w_up))
    return MOK_ERR_INVALID_ARG;
  SharedOperands sh{x_shared, s.T, w->ws_gate, w->ws_up, s.I_shared, a_shared};
  return launch_upgate_pair(xg, R, w->w_gate, w->w_up, offsets, s.E, R, s.D, s.I, a, st,
                            with_shared ? &sh : nullptr);
}

extern "C" mok_status mok_router(const mok_shape* shape, const void* x, const void* w_router, float* s_out,
                                 int32_t* topk_idx, float* g, void* stream) {
  if (!shape_ok(shape)) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  if (s.T == 0) return MOK_OK;
  if (s.E > 256) return MOK_ERR_UNSUPPORTED;
  if (!x || !w_router || !s_out || !topk_idx || !g || !aligned16(x) || !aligned16(w_router) || !aligned16(s_out))
    return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mok_status r = launch_router_pair(x, s.T, w_router, s.E, s.D, s_out, st);
  if (r != MOK_OK) return r;
  return launch_route(s_out, s.T, s.E, s.K, topk_idx, g, st);
}

extern "C" mok_status mok_expert_upgate_ring(const mok_shape* shape, const mok_weights* w, const void* x,
                                             const int32_t* table, const int32_t* offsets, void* a, void* ws,
                                             size_t ws_bytes, void* stream) {
  if (!shape_ok(shape) || !w) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  if (s.dtype != MOK_BF16) return MOK_ERR_UNSUPPORTED;
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  if (R == 0) return MOK_OK;
  if (!x || !table || !offsets || !a || !w->w_gate || !w->w_up || !aligned16(x) || !aligned16(a) ||
      !aligned16(w->w_gate) || !aligned16(w->w_up))
    return MOK_ERR_INVALID_ARG;
  const int64_t b = ring_chunk(s.chunk_rows);
  const size_t ring = round_up(ring_bytes(R, s.D, b));
  if (!ws || ws_bytes < ring + round_up(ring_counter_bytes(R, b)) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOK_ERR_WORKSPACE;
  return launch_upgate_ring(x, table, s.K, w->w_gate, w->w_up, offsets, s.E, R, s.D, s.I, a, ws,
                            ring_rows_for(R, b), static_cast<int>(b),
                            reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + ring),
                            static_cast<cudaStream_t>(stream));
}

extern "C" mok_status mok_expert_down(const mok_shape* shape, const mok_weights* w, const void* a,
                                      const uint8_t* a_scale, const int32_t* offsets, void* yg,
                                      const void* a_shared, void* ys, void* stream) {
  if (!shape_ok(shape) || !w) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  if (R == 0) return MOK_OK;
  const bool with_shared = s.I_shared > 0 && a_shared && ys;
  if (with_shared && (!w->ws_down || !aligned16(a_shared) || !aligned16(ys))) return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s.dtype == MOK_MXFP8) {
    if (!a || !a_scale || !offsets || !yg || !mx_weights_ok(w) || !aligned16(a) ||
        !aligned16(a_scale) || !aligned16(yg))
      return MOK_ERR_INVALID_ARG;
    mok_status r = launch_down_mx(a, a_scale, R, w->q_down, w->sc_down, offsets, s.E, s.D, s.I, yg, st);
    if (r != MOK_OK || !with_shared) return r;
    return launch_down(a_shared, s.T, w->ws_down, nullptr, 1, s.T, s.D, s.I_shared, ys, st);
  }
  if (!a || !offsets || !yg || !w->w_down || !aligned16(a) || !aligned16(yg) ||
      !aligned16(w->w_down))
    return MOK_ERR_INVALID_ARG;
  SharedOperands sh{a_shared, s.T, w->ws_down, nullptr, s.I_shared, ys};
  return launch_down_pair(a, R, w->w_down, offsets, s.E, R, s.D, s.I, yg, st, with_shared ? &sh : nullptr);
}

extern "C" mok_status mok_shared_ffn(const mok_shape* shape, const mok_weights* w, const void* x,
                                     void* ys, void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(shape) || !w) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  if (s.I_shared == 0 || s.T == 0) return MOK_OK;
  if (!x || !ys || !w->ws_gate || !w->ws_up || !w->ws_down || !aligned16(x) || !aligned16(ys))
    return MOK_ERR_INVALID_ARG;
  if (!ws || ws_bytes < static_cast<size_t>(s.T) * s.I_shared * 2) return MOK_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int sms = shared_expert_sms(s);
  mok_status r =
      launch_upgate(x, s.T, w->ws_gate, w->ws_up, nullptr, 1, s.T, s.D, s.I_shared, ws, st, sms);
  if (r != MOK_OK) return r;
  return launch_down(ws, s.T, w->ws_down, nullptr, 1, s.T, s.D, s.I_shared, ys, st, sms);
}

extern "C" mok_status mok_combine(const mok_shape* shape, const void* yg, const void* ys,
                                  const float* g, const int32_t* route_dst, void* out,
                                  void* stream) {
  if (!shape_ok(shape)) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  if (s.T == 0) return MOK_OK;
  if (!yg || !route_dst || !out || !aligned16(yg) || !aligned16(out) || (ys && !aligned16(ys)))
    return MOK_ERR_INVALID_ARG;
  return launch_combine(yg, ys, g, route_dst, s.T, s.K, s.D, out,
                        static_cast<cudaStream_t>(stream));
}

extern "C" mok_status mok_moe_fwd(const mok_shape* shape, const mok_weights* w, const void* x,
                                  const float* s_in, void* out, mok_plan_buf* saved, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (!shape_ok(shape) || !w) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  if (s.T == 0) return MOK_OK;
  const bool mx = s.dtype == MOK_MXFP8;
  if (!x || !s_in || !out || !aligned16(x) || !aligned16(out)) return MOK_ERR_INVALID_ARG;
  if (mx ? !mx_weights_ok(w) : (!w->w_gate || !w->w_up || !w->w_down)) return MOK_ERR_INVALID_ARG;
  if (s.I_shared && (!w->ws_gate || !w->ws_up || !w->ws_down)) return MOK_ERR_INVALID_ARG;
  const FwdLayout L = fwd_layout(s);
  if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOK_ERR_WORKSPACE;
  mok_plan_buf pb;
  if (saved) {
    pb = *saved;
    if (!pb.topk_idx || !pb.g || !pb.counts || !pb.offsets || !pb.table || !pb.route_dst)
      return MOK_ERR_INVALID_ARG;
  } else {
    pb.topk_idx = at<int32_t>(ws, L.topk);
    pb.g = at<float>(ws, L.g);
    pb.counts = at<int32_t>(ws, L.counts);
    pb.offsets = at<int32_t>(ws, L.offsets);
    pb.table = at<int32_t>(ws, L.table);
    pb.route_dst = at<int32_t>(ws, L.route_dst);
    pb.act = nullptr;
    pb.act_rows = 0;
    pb.act_shared = nullptr;
  }
  if (pb.act_rows < 0 || (pb.act && !aligned16(pb.act)) || (pb.act_shared && !aligned16(pb.act_shared)))
    return MOK_ERR_INVALID_ARG;
  // h, u of the groups that fit in the caller's store, kept for the backward
  const KeptAct kept{pb.act_rows > 0 ? pb.act : nullptr, pb.act_rows};
  const KeptAct kept_shared{s.I_shared ? pb.act_shared : nullptr, s.T};
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mok_status r;
  void* xg = at<void>(ws, L.xg);
  void* a = at<void>(ws, L.a);
  void* yg = at<void>(ws, L.yg);
  void* ys = s.I_shared ? at<void>(ws, L.ys) : nullptr;
  void* as = s.I_shared ? at<void>(ws, L.as) : nullptr;
  // The shared expert depends on x alone (paper note, "The production
  // details": it fills the first dispatch window).  Its up/gate (and for
  // MXFP8 its down projection) runs on a side stream next to route, plan and
  // dispatch (MXFP8: and the routed up/gate); the stream joins back before
  // the BF16 routed up/gate (whole-batch dispatch), else before the first
  // launch that reads its output.
  SideStream* side = nullptr;
  bool joined = true;
  // on an error after the fork, the caller's stream still waits for the side stream
  auto fail = [&](mok_status e) {
    if (!joined) cudaStreamWaitEvent(st, side->join, 0);
    return e;
  };
  if (s.I_shared) {
    if (!(side = side_stream())) return MOK_ERR_CUDA;
    if (cudaEventRecord(side->fork, st) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
      return MOK_ERR_CUDA;
    const int sms = shared_expert_sms(s);
    r = launch_upgate(x, s.T, w->ws_gate, w->ws_up, nullptr, 1, s.T, s.D, s.I_shared, as, side->s, sms,
                      kept_shared);
    if (r == MOK_OK && mx)
      r = launch_down(as, s.T, w->ws_down, nullptr, 1, s.T, s.D, s.I_shared, ys, side->s, sms);
    if (cudaEventRecord(side->join, side->s) != cudaSuccess) return MOK_ERR_CUDA;
    joined = false;
    if (r != MOK_OK) return fail(r);
  }
  if ((r = launch_route(s_in, s.T, s.E, s.K, pb.topk_idx, pb.g, st)) != MOK_OK) return fail(r);
  if ((r = launch_plan(pb.topk_idx, R, s.E, pb.counts, pb.offsets, pb.table, pb.route_dst,
                       at<int>(ws, L.hist), st)) != MOK_OK)
    return fail(r);
  if (mx) {
    void* asc = at<void>(ws, L.a_scale);
    if (uses_ring(s)) {
      // the quantising dispatch runs inside the up/gate launch, through the ring in xg
      const int64_t b = ring_chunk(s.chunk_rows);
      if ((r = launch_upgate_mx_ring(x, pb.table, s.K, w->q_gate, w->sc_gate, w->q_up, w->sc_up, pb.offsets, s.E, R,
                                     s.D, s.I, a, asc, at<void>(ws, L.xg_scale), xg, ring_rows_for(R, b),
                                     static_cast<int>(b), at<int32_t>(ws, L.ring_counters), st, kept)) != MOK_OK)
        return fail(r);
    } else {
      if ((r = launch_dispatch_mxfp8(x, pb.route_dst, pb.table, pb.offsets, s.T, s.K, s.D, s.E, xg,
                                     at<uint8_t>(ws, L.xg_scale), st)) != MOK_OK)
        return fail(r);
      if ((r = launch_upgate_mx(xg, at<void>(ws, L.xg_scale), R, w->q_gate, w->sc_gate, w->q_up,
                                w->sc_up, pb.offsets, s.E, s.D, s.I, a, asc, st, kept, w->sc_gu_pair)) != MOK_OK)
        return fail(r);
    }
    if ((r = launch_down_mx(a, asc, R, w->q_down, w->sc_down, pb.offsets, s.E, s.D, s.I, yg, st)) !=
        MOK_OK)
      return fail(r);
  } else {
    if (uses_ring(s)) {
      // the dispatch runs inside the up/gate launch, through the ring in xg
      const int64_t b = ring_chunk(s.chunk_rows);
      if ((r = launch_upgate_ring(x, pb.table, s.K, w->w_gate, w->w_up, pb.offsets, s.E, R, s.D, s.I, a, xg,
                                  ring_rows_for(R, b), static_cast<int>(b), at<int32_t>(ws, L.ring_counters),
                                  st, kept)) != MOK_OK)
        return fail(r);
    } else {
      if ((r = launch_dispatch_bf16(x, pb.route_dst, s.T, s.K, s.D, xg, nullptr, nullptr, st)) != MOK_OK)
        return fail(r);
      // The shared up/gate ran beside route, plan and the dispatch (its
      // kernel leaves them room on every SM); the routed up/gate starts once
      // it is done, on the whole GPU, instead of queueing its CTAs behind
      // the shared expert's tail.
      if (!joined) {
        joined = true;
        if (cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return MOK_ERR_CUDA;
      }
      if ((r = launch_upgate_pair(xg, R, w->w_gate, w->w_up, pb.offsets, s.E, R, s.D, s.I, a, st, nullptr,
                                  kept)) != MOK_OK)
        return fail(r);
    }
  }
  if (!joined) {
    joined = true;
    if (cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return MOK_ERR_CUDA;
  }
  if (!mx) {
    // the shared expert's down tiles run inside the routed down launch
    SharedOperands sh_dn{as, s.T, w->ws_down, nullptr, s.I_shared, ys};
    if ((r = launch_down_pair(a, R, w->w_down, pb.offsets, s.E, R, s.D, s.I, yg, st,
                              s.I_shared ? &sh_dn : nullptr)) != MOK_OK)
      return r;
  }
  return launch_combine(yg, ys, pb.g, pb.route_dst, s.T, s.K, s.D, out, st);
}

extern "C" size_t mok_mxfp8_scale_bytes(int64_t rows, int64_t cols, int32_t groups) {
  if (rows < 0 || cols <= 0 || cols % 128 || groups < 0) return 0;
  return mx_scale_bytes(rows, cols, groups);
}

extern "C" mok_status mok_quantize_mxfp8(const void* src, int64_t rows, int64_t cols, void* q,
                                         uint8_t* scale, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 128) return MOK_ERR_INVALID_ARG;
  if (rows == 0) return MOK_OK;
  if (!src || !q || !scale || !aligned16(src) || !aligned16(q)) return MOK_ERR_INVALID_ARG;
  return launch_quantize_mxfp8(src, rows, cols, q, scale, static_cast<cudaStream_t>(stream));
}

extern "C" mok_status mok_mxfp8_pair_scales(const mok_shape* shape, const mok_weights* w, uint8_t* sc_gu_pair,
                                            void* stream) {
  if (!shape_ok(shape) || !w) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  if (!w->sc_gate || !w->sc_up || !sc_gu_pair || !aligned16(w->sc_gate) || !aligned16(w->sc_up) ||
      !aligned16(sc_gu_pair))
    return MOK_ERR_INVALID_ARG;
  return launch_pair_scales(w->sc_gate, w->sc_up, s.E, s.I, s.D, sc_gu_pair, static_cast<cudaStream_t>(stream));
}

extern "C" mok_status mok_quantize_mxfp8_bwd_weights(const mok_shape* shape, const mok_weights* w, void* qt_down,
                                                     uint8_t* sct_down, void* qt_gu, uint8_t* sct_gu, void* stream) {
  if (!shape_ok(shape) || !w) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  if (s.D % 128 || s.I % 128) return MOK_ERR_INVALID_ARG;
  if (!w->w_gate || !w->w_up || !w->w_down || !qt_down || !sct_down || !qt_gu || !sct_gu ||
      !aligned16(w->w_gate) || !aligned16(w->w_up) || !aligned16(w->w_down) || !aligned16(qt_down) ||
      !aligned16(sct_down) || !aligned16(qt_gu) || !aligned16(sct_gu))
    return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  mok_status r;
  // W_down [E][D][I]: output rows (e, i), D values each
  if ((r = launch_quantize_cols_mxfp8(w->w_down, s.E, s.D, s.I, qt_down, sct_down, s.D, 0, st)) != MOK_OK) return r;
  // W_gate, W_up [E][I][D]: output rows (e, d), I values each, side by side
  if ((r = launch_quantize_cols_mxfp8(w->w_gate, s.E, s.I, s.D, qt_gu, sct_gu, 2 * s.I, 0, st)) != MOK_OK) return r;
  return launch_quantize_cols_mxfp8(w->w_up, s.E, s.I, s.D, qt_gu, sct_gu, 2 * s.I, s.I, st);
}

extern "C" int32_t mok_bwd_shared_sms(const mok_shape* shape) {
  if (!shape_ok(shape)) return -1;
  return bwd_shared_split(*shape);
}

extern "C" mok_status mok_moe_bwd(const mok_shape* shape, const mok_weights* w, const void* x,
                                  const float* s_in, const mok_plan_buf* saved, const void* dy,
                                  void* dx, void* dw_gate, void* dw_up, void* dw_down,
                                  void* dws_gate, void* dws_up, void* dws_down, float* ds,
                                  float* dg, void* ws, size_t ws_bytes, void* stream) {
  if (!shape_ok(shape) || !w || !saved) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = *shape;
  const bool mx = s.dtype == MOK_MXFP8;
  if (mx && (!mx_weights_ok(w) || !mx_bwd_weights_ok(w))) return MOK_ERR_INVALID_ARG;
  if (mx && (s.I % 256 || s.D % 256)) return MOK_ERR_UNSUPPORTED;  // 256-column tiles of t and dX
  if (s.T == 0) return MOK_OK;
  const mok_plan_buf& pb = *saved;
  if (!x || !s_in || !dy || !dx || !dw_gate || !dw_up || !dw_down || !ds || !pb.topk_idx ||
      !pb.g || !pb.offsets || !pb.table || !pb.route_dst || !w->w_gate || !w->w_up || !w->w_down)
    return MOK_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(dw_gate) ||
      !aligned16(dw_up) || !aligned16(dw_down) || !aligned16(w->w_gate) || !aligned16(w->w_up) ||
      !aligned16(w->w_down))
    return MOK_ERR_INVALID_ARG;
  if (s.I_shared && (!w->ws_gate || !w->ws_up || !w->ws_down || !dws_gate || !dws_up || !dws_down))
    return MOK_ERR_INVALID_ARG;
  if (pb.act_rows < 0 || (pb.act && !aligned16(pb.act)) || (pb.act_shared && !aligned16(pb.act_shared)))
    return MOK_ERR_INVALID_ARG;
  const BwdLayout L = bwd_layout(s);
  if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOK_ERR_WORKSPACE;
  const int64_t R = static_cast<int64_t>(s.T) * s.K;
  // the groups whose h, u the forward kept (rows below kept_rows) skip the
  // replay; with every row kept no replay runs at all
  const KeptAct kept{pb.act_rows > 0 ? pb.act : nullptr, pb.act_rows};
  const int32_t kept_rows = kept.limit();
  const bool replay = kept_rows < R;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* xg = at<void>(ws, L.xg);
  void* dyg = at<void>(ws, L.dyg);
  float* g_route = at<float>(ws, L.g_route);
  void* dh = at<void>(ws, L.dh);
  void* du = at<void>(ws, L.du);
  void* ag = at<void>(ws, L.ag);
  float* dgp = at<float>(ws, L.dgp);
  void* dxr = at<void>(ws, L.dxr);
  mok_status r;
  // The shared expert's backward (paper note, "The production details": the
  // shared expert needs no dispatch) reads x, dY and its own weights only.
  // With shape.bwd_shared_sms it runs on a side stream on `ksh` SMs while
  // the routed dgrad and dX run on the rest, and the caller's stream joins
  // it before the reverse combine, the first launch that reads its dX;
  // without (the default, faster on a GB300: the routed dgrad and dX need
  // every SM for their bandwidth) it runs after the routed dX.
  const int ksh = bwd_shared_split(s);
  const int routed_sms = ksh > 0 ? num_sms() - ksh : 0;
  void* dxs = s.I_shared ? at<void>(ws, L.dxs) : nullptr;
  auto shared_bwd = [&](cudaStream_t ss, int sms) -> mok_status {
    void* dhs = at<void>(ws, L.dhs);
    void* dus = at<void>(ws, L.dus);
    void* ags = at<void>(ws, L.ags);
    mok_status e;
    // h, u from the forward's store when it kept them, else replayed from x
    if (pb.act_shared) {
      if ((e = launch_bwd_dgrad_kept(dy, s.T, w->ws_down, nullptr, 1, s.D, s.I_shared, nullptr, pb.act_shared, s.T,
                                     dhs, dus, ags, nullptr, ss, sms)) != MOK_OK)
        return e;
    } else if ((e = launch_bwd_dgrad(x, dy, s.T, w->ws_gate, w->ws_up, w->ws_down, nullptr, 1, s.D, s.I_shared,
                                     nullptr, dhs, dus, ags, nullptr, ss, 0, sms)) != MOK_OK) {
      return e;
    }
    if ((e = launch_bwd_dx(dhs, dus, s.T, w->ws_gate, w->ws_up, nullptr, 1, s.D, s.I_shared, dxs, ss, sms)) !=
        MOK_OK)
      return e;
    if ((e = launch_wgrad(dy, ags, s.T, nullptr, 1, s.D, s.I_shared, dws_down, ss, sms)) != MOK_OK) return e;
    if ((e = launch_wgrad(dhs, x, s.T, nullptr, 1, s.I_shared, s.D, dws_gate, ss, sms)) != MOK_OK) return e;
    return launch_wgrad(dus, x, s.T, nullptr, 1, s.I_shared, s.D, dws_up, ss, sms);
  };
  SideStream* side = nullptr;
  bool joined = true;
  // on an error after the fork, the caller's stream still waits for the side stream
  auto fail = [&](mok_status e) {
    if (!joined) cudaStreamWaitEvent(st, side->join, 0);
    return e;
  };
  if (ksh > 0) {
    if (!(side = side_stream())) return MOK_ERR_CUDA;
    if (cudaEventRecord(side->fork, st) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
      return MOK_ERR_CUDA;
    r = shared_bwd(side->s, ksh);
    if (cudaEventRecord(side->join, side->s) != cudaSuccess) return MOK_ERR_CUDA;
    joined = false;
    if (r != MOK_OK) return fail(r);
  }
  // gather x, dY and the route weights into expert order (the forward's plan)
  if ((r = launch_dispatch_bf16(x, pb.route_dst, s.T, s.K, s.D, xg, pb.g, g_route, st)) != MOK_OK) return fail(r);
  if ((r = launch_dispatch_bf16(dy, pb.route_dst, s.T, s.K, s.D, dyg, nullptr, nullptr, st)) != MOK_OK)
    return fail(r);
  if (mx) {
    // MXFP8: quantising dispatches of x and dY; replay h, u; t = dY W_down
    // (W_down^T quantised along D); the activation gradient with [dh | du]
    // quantised along 2I; dX routes = [dh | du] [W_gate ; W_up]
    void* xq = at<void>(ws, L.xq);
    uint8_t* xq_sc = at<uint8_t>(ws, L.xq_sc);
    void* dyq = at<void>(ws, L.dyq);
    uint8_t* dyq_sc = at<uint8_t>(ws, L.dyq_sc);
    void* hh = at<void>(ws, L.hh);
    void* uu = at<void>(ws, L.uu);
    void* tt = at<void>(ws, L.tt);
    void* dhu_q = at<void>(ws, L.dhu_q);
    uint8_t* dhu_sc = at<uint8_t>(ws, L.dhu_sc);
    if (replay && (r = launch_dispatch_mxfp8(x, pb.route_dst, pb.table, pb.offsets, s.T, s.K, s.D, s.E, xq,
                                             xq_sc, st)) != MOK_OK)
      return fail(r);
    if ((r = launch_dispatch_mxfp8(dy, pb.route_dst, pb.table, pb.offsets, s.T, s.K, s.D, s.E, dyq, dyq_sc, st)) !=
        MOK_OK)
      return fail(r);
    if (replay && (r = launch_replay_mx(xq, xq_sc, R, w->q_gate, w->sc_gate, w->q_up, w->sc_up, pb.offsets, s.E,
                                        s.D, s.I, hh, uu, st, kept_rows)) != MOK_OK)
      return fail(r);
    if ((r = launch_down_mx(dyq, dyq_sc, R, w->qt_down, w->sct_down, pb.offsets, s.E, s.I, s.D, tt, st,
                            /*f32_out=*/true, routed_sms)) != MOK_OK)
      return fail(r);
    if ((r = launch_act_grad_mx(hh, uu, tt, g_route, pb.table, pb.offsets, R, s.I, s.E, dh, du, ag, dhu_q, dhu_sc,
                                dgp, st, kept)) != MOK_OK)
      return fail(r);
    if ((r = launch_down_mx(dhu_q, dhu_sc, R, w->qt_gu, w->sct_gu, pb.offsets, s.E, s.D, 2 * s.I, dxr, st,
                            /*f32_out=*/false, routed_sms)) != MOK_OK)
      return fail(r);
  } else {
    // t = dY W_down with the kept h, u; replay h, u for the other groups;
    // dh, du, g*a, <t, a> partials
    if (kept_rows > 0 && (r = launch_bwd_dgrad_kept(dyg, R, w->w_down, pb.offsets, s.E, s.D, s.I, g_route,
                                                    kept.act, kept_rows, dh, du, ag, dgp, st, routed_sms)) != MOK_OK)
      return fail(r);
    if (replay && (r = launch_bwd_dgrad(xg, dyg, R, w->w_gate, w->w_up, w->w_down, pb.offsets, s.E, s.D, s.I,
                                        g_route, dh, du, ag, dgp, st, kept_rows, routed_sms)) != MOK_OK)
      return fail(r);
    if ((r = launch_bwd_dx(dh, du, R, w->w_gate, w->w_up, pb.offsets, s.E, s.D, s.I, dxr, st, routed_sms)) !=
        MOK_OK)
      return fail(r);
  }
  if (s.I_shared && ksh == 0 && (r = shared_bwd(st, 0)) != MOK_OK) return r;
  if (!joined) {
    joined = true;
    if (cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return MOK_ERR_CUDA;
  }
  // reverse combine in fixed k order
  if ((r = launch_combine(dxr, dxs, nullptr, pb.route_dst, s.T, s.K, s.D, dx, st)) != MOK_OK) return r;
  // per-expert weight gradients, K over the expert's rows
  if ((r = launch_wgrad(dyg, ag, R, pb.offsets, s.E, s.D, s.I, dw_down, st)) != MOK_OK) return r;
  if ((r = launch_wgrad(dh, xg, R, pb.offsets, s.E, s.I, s.D, dw_gate, st)) != MOK_OK) return r;
  if ((r = launch_wgrad(du, xg, R, pb.offsets, s.E, s.I, s.D, dw_up, st)) != MOK_OK) return r;
  return launch_router_grad(dgp, mx ? 1 : s.I / 32, pb.route_dst, pb.topk_idx, pb.g, s_in, s.T, s.E, s.K,
                            ds, dg, st);
}
