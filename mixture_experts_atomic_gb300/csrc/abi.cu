// extern "C" entry points of the moeblaze library (declared in
// include/moeblaze.h): argument validation, scratch carving and the order of
// the stages; every stage runs in the kernels of dispatch.cu, identity.cu,
// simt.cu, gemm_tc.cu and router.cu.
#include <atomic>
#include <cstring>

#include "common.cuh"

namespace moeblaze {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {
std::atomic<int64_t> g_launches{0};
thread_local void** g_events = nullptr;
thread_local int32_t g_nevents = 0;
thread_local uint64_t g_wait_ns = 0;
thread_local int g_withhold = 0;
}  // namespace

void fault_injection(uint64_t* wait_ns, int* withhold) {
  *wait_ns = g_wait_ns;
  *withhold = g_withhold;
}

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

void stage_event(int i, cudaStream_t st) {
  if (g_events && i < g_nevents && g_events[i]) cudaEventRecord(reinterpret_cast<cudaEvent_t>(g_events[i]), st);
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// shape checks shared by every entry point
moeblaze_status check_shape(const moeblaze_shape* s) {
  if (!s) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->L < 0 || s->E < 1 || s->K < 1 || s->d < 1) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->K > s->E) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->dtype != MOEBLAZE_F32 && s->dtype != MOEBLAZE_BF16) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->act != MOEBLAZE_SWIGLU && s->act != MOEBLAZE_SILU && s->act != MOEBLAZE_IDENTITY)
    return MOEBLAZE_ERR_INVALID_ARG;
  if (s->act != MOEBLAZE_IDENTITY && s->h < 1) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->flags & ~MOEBLAZE_RECOMPUTE_H) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->E > kMaxE || s->K > kMaxK) return MOEBLAZE_ERR_UNSUPPORTED;
  if (s->L * (int64_t)s->K + (int64_t)s->E * kRowPad >= (int64_t(1) << 31)) return MOEBLAZE_ERR_UNSUPPORTED;
  if (s->act == MOEBLAZE_IDENTITY) {
    if (s->d % (s->dtype == MOEBLAZE_BF16 ? 8 : 4) != 0) return MOEBLAZE_ERR_UNSUPPORTED;
  } else if (s->dtype == MOEBLAZE_BF16) {
    if (s->d % 128 != 0 || s->h % 128 != 0) return MOEBLAZE_ERR_UNSUPPORTED;
  } else {
    if (s->d % 4 != 0 || s->h % 4 != 0) return MOEBLAZE_ERR_UNSUPPORTED;
  }
  return MOEBLAZE_OK;
}

moeblaze_status check_dispatch(const moeblaze_dispatch* d) {
  if (!d) return MOEBLAZE_ERR_INVALID_ARG;
  const void* ps[5] = {d->expert_token_indices, d->expert_token_offsets, d->token_expert_indices, d->token_index_map,
                       d->meta};
  for (const void* p : ps)
    if (!p || !aligned16(p)) return MOEBLAZE_ERR_INVALID_ARG;
  return MOEBLAZE_OK;
}

bool ok_ptr(const void* p) { return p && aligned16(p); }
bool ok_ptr4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// shape checks of the router entry points (h and act are not used)
moeblaze_status check_router_shape(const moeblaze_shape* s) {
  if (!s) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->L < 0 || s->E < 1 || s->K < 1 || s->d < 1 || s->K > s->E) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->dtype != MOEBLAZE_F32 && s->dtype != MOEBLAZE_BF16) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->E > kMaxRouterE || s->K > kMaxK || s->d % 64 != 0) return MOEBLAZE_ERR_UNSUPPORTED;
  if (s->L * (int64_t)s->K >= (int64_t(1) << 31)) return MOEBLAZE_ERR_UNSUPPORTED;
  return MOEBLAZE_OK;
}

size_t elem(const moeblaze_shape* s) { return s->dtype == MOEBLAZE_BF16 ? 2 : 4; }
int nbranch(const moeblaze_shape* s) { return s->act == MOEBLAZE_SWIGLU ? 2 : 1; }

// MOEBLAZE_RECOMPUTE_H applies to the bf16 expert layers: H and Hg are then
// recomputed from the saved A, B inside the down-projection and dW3 GEMMs
// and never stored.
bool recompute_h(const moeblaze_shape* s) {
  return s->dtype == MOEBLAZE_BF16 && s->act != MOEBLAZE_IDENTITY && (s->flags & MOEBLAZE_RECOMPUTE_H);
}

// saved:            A | B (SwiGLU) (rows x h each); bf16 with recompute: | one fp32 gate per row
// forward scratch:  H (rows x h; not when recomputed) | y32 (L x d fp32) + tile counters (bf16 only)
// backward scratch: bf16: Hg (rows x h; not when recomputed) | dX32 (L x d fp32) + tile counters
//                   (dA, dB overwrite the saved A, B);  fp32: dAB (rows x nb*h) | Hg (rows x h)
size_t fwd_ws(const moeblaze_shape* s) {
  if (s->act == MOEBLAZE_IDENTITY) return 0;
  const int64_t rows = max_padded_rows(s->L * s->K, s->E);
  size_t b = recompute_h(s) ? 0 : align_up((size_t)rows * s->h * elem(s), 256);
  if (s->dtype == MOEBLAZE_BF16) b += align_up((size_t)s->L * s->d * 4, 256) + kSchedBytes;
  return b;
}
size_t hg_bytes(const moeblaze_shape* s) {
  const int64_t rows = max_padded_rows(s->L * s->K, s->E);
  return recompute_h(s) ? 0 : align_up((size_t)rows * s->h * elem(s), 256);
}
size_t bwd_ws(const moeblaze_shape* s) {
  if (s->act == MOEBLAZE_IDENTITY) return 0;
  const int64_t rows = max_padded_rows(s->L * s->K, s->E);
  if (s->dtype == MOEBLAZE_BF16) return hg_bytes(s) + align_up((size_t)s->L * s->d * 4, 256) + kSchedBytes;
  return align_up((size_t)rows * nbranch(s) * s->h * elem(s), 256) + hg_bytes(s);
}

moeblaze_status zero_weight_grads(const moeblaze_shape* s, void* dW1, void* dW2, void* dW3, cudaStream_t st) {
  const size_t n = (size_t)s->E * s->d * s->h * elem(s);
  MB_CUDA(cudaMemsetAsync(dW1, 0, n, st));
  if (dW2) MB_CUDA(cudaMemsetAsync(dW2, 0, n, st));
  MB_CUDA(cudaMemsetAsync(dW3, 0, n, st));
  return MOEBLAZE_OK;
}

}  // namespace
}  // namespace moeblaze

using namespace moeblaze;

extern "C" {

int32_t moeblaze_version(void) { return 10000; }

void moeblaze_set_stage_events(void** events, int32_t n) {
  g_events = events;
  g_nevents = events ? n : 0;
}

int64_t moeblaze_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

void moeblaze_set_fault_injection(int64_t wait_limit_ns, int32_t withhold) {
  g_wait_ns = wait_limit_ns > 0 ? (uint64_t)wait_limit_ns : 0;
  g_withhold = withhold ? 1 : 0;
}

const char* moeblaze_status_string(moeblaze_status st) {
  switch (st) {
    case MOEBLAZE_OK: return "ok";
    case MOEBLAZE_ERR_INVALID_ARG: return "invalid argument";
    case MOEBLAZE_ERR_UNSUPPORTED: return "unsupported shape or type";
    case MOEBLAZE_ERR_BAD_ROUTING: return "bad routing: expert id out of range or repeated within a token";
    case MOEBLAZE_ERR_WORKSPACE: return "workspace too small";
    case MOEBLAZE_ERR_TIMEOUT: return "a device-side wait timed out";
    case MOEBLAZE_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

size_t moeblaze_dispatch_meta_bytes(const moeblaze_shape* s) {
  if (check_shape(s) != MOEBLAZE_OK) return 0;
  return meta_bytes(s->L * s->K, s->E);
}

size_t moeblaze_dispatch_workspace_bytes(const moeblaze_shape* s) {
  if (check_shape(s) != MOEBLAZE_OK) return 0;
  return dispatch_ws_bytes(*s);
}

size_t moeblaze_saved_bytes(const moeblaze_shape* s) {
  if (check_shape(s) != MOEBLAZE_OK || s->act == MOEBLAZE_IDENTITY) return 0;
  const int64_t rows = max_padded_rows(s->L * s->K, s->E);
  return (size_t)rows * nbranch(s) * s->h * elem(s) + (recompute_h(s) ? (size_t)rows * 4 : 0);
}

size_t moeblaze_forward_workspace_bytes(const moeblaze_shape* s) {
  if (check_shape(s) != MOEBLAZE_OK) return 0;
  return fwd_ws(s);
}

size_t moeblaze_backward_workspace_bytes(const moeblaze_shape* s) {
  if (check_shape(s) != MOEBLAZE_OK) return 0;
  return bwd_ws(s);
}

moeblaze_status moeblaze_dispatch_build(const moeblaze_shape* s, const int32_t* topk_ids,
                                        const moeblaze_dispatch* out, void* ws, size_t ws_bytes, int validate,
                                        moeblaze_stream stream) {
  moeblaze_status r = check_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if ((r = check_dispatch(out)) != MOEBLAZE_OK) return r;
  if (s->L > 0 && !ok_ptr(topk_ids)) return MOEBLAZE_ERR_INVALID_ARG;
  if (ws_bytes < dispatch_ws_bytes(*s)) return MOEBLAZE_ERR_WORKSPACE;
  if (!ok_ptr(ws)) return MOEBLAZE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  r = launch_dispatch(*s, topk_ids, *out, ws, st);
  if (r != MOEBLAZE_OK || !validate) return r;
  int32_t code = 0;
  MB_CUDA(cudaMemcpyAsync(&code, out->meta, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  MB_CUDA(cudaStreamSynchronize(st));
  return (code & kErrBadRouting) ? MOEBLAZE_ERR_BAD_ROUTING : MOEBLAZE_OK;
}

moeblaze_status moeblaze_dispatch_build_static(const moeblaze_shape* s, const int32_t* topk_ids,
                                               const moeblaze_dispatch* out, int validate, moeblaze_stream stream) {
  moeblaze_status r = check_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if ((r = check_dispatch(out)) != MOEBLAZE_OK) return r;
  if (s->L > 0 && !ok_ptr(topk_ids)) return MOEBLAZE_ERR_INVALID_ARG;
  if (dispatch_ws_bytes(*s) > MOEBLAZE_STATIC_SCRATCH_BYTES) return MOEBLAZE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  r = launch_dispatch_static(*s, topk_ids, *out, st);
  if (r != MOEBLAZE_OK || !validate) return r;
  int32_t code = 0;
  MB_CUDA(cudaMemcpyAsync(&code, out->meta, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  MB_CUDA(cudaStreamSynchronize(st));
  return (code & kErrBadRouting) ? MOEBLAZE_ERR_BAD_ROUTING : MOEBLAZE_OK;
}

moeblaze_status moeblaze_forward(const moeblaze_shape* s, const void* x, const float* gates,
                                 const moeblaze_dispatch* disp, const void* W1, const void* W2, const void* W3,
                                 void* y, void* saved, void* ws, size_t ws_bytes, moeblaze_stream stream) {
  moeblaze_status r = check_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if ((r = check_dispatch(disp)) != MOEBLAZE_OK) return r;
  // token-sized buffers may be empty (NULL) when L == 0
  const bool tok_ok = s->L == 0 || (ok_ptr(x) && ok_ptr(gates) && ok_ptr(y));
  if (!tok_ok) return MOEBLAZE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (s->act == MOEBLAZE_IDENTITY) return launch_identity_combine(*s, x, *disp, gates, y, st);
  const bool sw = s->act == MOEBLAZE_SWIGLU;
  if (!ok_ptr(W1) || !ok_ptr(W3) || (sw && !ok_ptr(W2)) || !ok_ptr(saved)) return MOEBLAZE_ERR_INVALID_ARG;
  if (ws_bytes < fwd_ws(s)) return MOEBLAZE_ERR_WORKSPACE;
  if (!ok_ptr(ws)) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->L == 0) return MOEBLAZE_OK;
  const int64_t rows = max_padded_rows(s->L * s->K, s->E);
  char* w = reinterpret_cast<char*>(ws);
  if (s->dtype == MOEBLAZE_F32) {
    return simt_forward(*s, (const float*)x, gates, *disp, (const float*)W1, sw ? (const float*)W2 : nullptr,
                        (const float*)W3, (float*)y, (float*)saved, (float*)w, st);
  }
  const size_t hb = recompute_h(s) ? 0 : align_up((size_t)rows * s->h * 2, 256);
  __nv_bfloat16* H = hb ? reinterpret_cast<__nv_bfloat16*>(w) : nullptr;
  return tc_forward(*s, (const __nv_bfloat16*)x, gates, *disp, (const __nv_bfloat16*)W1,
                    sw ? (const __nv_bfloat16*)W2 : nullptr, (const __nv_bfloat16*)W3, (__nv_bfloat16*)y,
                    (__nv_bfloat16*)saved, H, reinterpret_cast<float*>(w + hb), st);
}

moeblaze_status moeblaze_backward(const moeblaze_shape* s, const void* dY, const void* x, const float* gates,
                                  const moeblaze_dispatch* disp, const void* W1, const void* W2, const void* W3,
                                  void* saved, void* dX, void* dW1, void* dW2, void* dW3, float* dgates,
                                  void* ws, size_t ws_bytes, moeblaze_stream stream) {
  moeblaze_status r = check_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if ((r = check_dispatch(disp)) != MOEBLAZE_OK) return r;
  const bool tok_ok = s->L == 0 || (ok_ptr(dY) && ok_ptr(gates) && ok_ptr(dX) && ok_ptr(x));
  if (!tok_ok) return MOEBLAZE_ERR_INVALID_ARG;
  if (dgates && !aligned16(dgates)) return MOEBLAZE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (s->act == MOEBLAZE_IDENTITY) {
    r = launch_identity_combine(*s, dY, *disp, gates, dX, st);
    if (r != MOEBLAZE_OK || !dgates) return r;
    return launch_identity_dgates(*s, x, dY, dgates, st);
  }
  const bool sw = s->act == MOEBLAZE_SWIGLU;
  if (!ok_ptr(W1) || !ok_ptr(W3) || (sw && !ok_ptr(W2)) || !ok_ptr(saved)) return MOEBLAZE_ERR_INVALID_ARG;
  if (!ok_ptr(dW1) || !ok_ptr(dW3) || (sw && !ok_ptr(dW2))) return MOEBLAZE_ERR_INVALID_ARG;
  if (ws_bytes < bwd_ws(s)) return MOEBLAZE_ERR_WORKSPACE;
  if (!ok_ptr(ws)) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->L == 0) return zero_weight_grads(s, dW1, sw ? dW2 : nullptr, dW3, st);
  if (dgates) MB_CUDA(cudaMemsetAsync(dgates, 0, sizeof(float) * s->L * s->K, st));
  const int64_t rows = max_padded_rows(s->L * s->K, s->E);
  char* w = reinterpret_cast<char*>(ws);
  const size_t es = elem(s);
  if (s->dtype == MOEBLAZE_F32) {
    char* dAB = w;
    char* Hg = w + align_up((size_t)rows * nbranch(s) * s->h * es, 256);
    return simt_backward(*s, (const float*)dY, (const float*)x, gates, *disp, (const float*)W1,
                         sw ? (const float*)W2 : nullptr, (const float*)W3, (const float*)saved, (float*)dX,
                         (float*)dW1, sw ? (float*)dW2 : nullptr, (float*)dW3, dgates, (float*)dAB, (float*)Hg, st);
  }
  // bf16: Hg (not when recomputed) | dX32; dA, dB go over the saved A, B
  char* dX32 = w + hg_bytes(s);
  return tc_backward(*s, (const __nv_bfloat16*)dY, (const __nv_bfloat16*)x, gates, *disp, (const __nv_bfloat16*)W1,
                     sw ? (const __nv_bfloat16*)W2 : nullptr, (const __nv_bfloat16*)W3, (__nv_bfloat16*)saved,
                     (__nv_bfloat16*)dX, (__nv_bfloat16*)dW1, sw ? (__nv_bfloat16*)dW2 : nullptr, (__nv_bfloat16*)dW3,
                     dgates, recompute_h(s) ? nullptr : (__nv_bfloat16*)w, (float*)dX32, st);
}

moeblaze_status moeblaze_device_error(const moeblaze_shape* s, const moeblaze_dispatch* disp, int32_t* code,
                                      moeblaze_stream stream) {
  moeblaze_status r = check_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if (!disp || !ok_ptr(disp->meta) || !code) return MOEBLAZE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t c = 0;
  MB_CUDA(cudaMemcpyAsync(&c, disp->meta, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  MB_CUDA(cudaStreamSynchronize(st));
  *code = c;
  if (c & kErrBadRouting) return MOEBLAZE_ERR_BAD_ROUTING;
  if (c & kErrTimeout) return MOEBLAZE_ERR_TIMEOUT;
  if (c & kErrShapeMismatch) return MOEBLAZE_ERR_INVALID_ARG;
  return MOEBLAZE_OK;
}

moeblaze_status moeblaze_dispatch_meta_check(const moeblaze_shape* s, const void* meta_header) {
  moeblaze_status r = check_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if (!meta_header) return MOEBLAZE_ERR_INVALID_ARG;
  return meta_matches(reinterpret_cast<const int32_t*>(meta_header), s->L, s->E, s->K) ? MOEBLAZE_OK
                                                                                     : MOEBLAZE_ERR_INVALID_ARG;
}

size_t moeblaze_router_backward_workspace_bytes(const moeblaze_shape* s) {
  if (check_router_shape(s) != MOEBLAZE_OK) return 0;
  return router_ws_bytes(*s);
}

moeblaze_status moeblaze_router_forward(const moeblaze_shape* s, const void* x, const float* Wr, const float* bias,
                                        int32_t* topk_ids, float* gates, moeblaze_stream stream) {
  moeblaze_status r = check_router_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if (!ok_ptr4(Wr) || (bias && !ok_ptr4(bias))) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->L > 0 && (!ok_ptr(x) || !ok_ptr4(topk_ids) || !ok_ptr4(gates))) return MOEBLAZE_ERR_INVALID_ARG;
  return launch_router_forward(*s, x, Wr, bias, topk_ids, gates, reinterpret_cast<cudaStream_t>(stream));
}

size_t moeblaze_router_dispatch_workspace_bytes(const moeblaze_shape* s) {
  if (check_shape(s) != MOEBLAZE_OK || check_router_shape(s) != MOEBLAZE_OK) return 0;
  return router_dispatch_fused(*s) ? router_dispatch_ws_bytes(*s) : dispatch_ws_bytes(*s);
}

moeblaze_status moeblaze_router_dispatch_build(const moeblaze_shape* s, const void* x, const float* Wr,
                                               const float* bias, int32_t* topk_ids, float* gates,
                                               const moeblaze_dispatch* out, void* ws, size_t ws_bytes,
                                               moeblaze_stream stream) {
  moeblaze_status r = check_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if ((r = check_router_shape(s)) != MOEBLAZE_OK) return r;
  if ((r = check_dispatch(out)) != MOEBLAZE_OK) return r;
  if (!ok_ptr4(Wr) || (bias && !ok_ptr4(bias))) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->L > 0 && (!ok_ptr(x) || !ok_ptr4(topk_ids) || !ok_ptr4(gates))) return MOEBLAZE_ERR_INVALID_ARG;
  if (ws_bytes < moeblaze_router_dispatch_workspace_bytes(s)) return MOEBLAZE_ERR_WORKSPACE;
  if (!ok_ptr(ws)) return MOEBLAZE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (router_dispatch_fused(*s)) return launch_router_dispatch(*s, x, Wr, bias, topk_ids, gates, *out, ws, st);
  // shapes the fused kernel does not take (fp32 x, more than 64 experts, no
  // tokens): the router, then the dispatch build on its ids
  if (s->L > 0 && (r = launch_router_forward(*s, x, Wr, bias, topk_ids, gates, st)) != MOEBLAZE_OK) return r;
  return launch_dispatch(*s, topk_ids, *out, ws, st);
}

moeblaze_status moeblaze_router_backward(const moeblaze_shape* s, const void* x, const float* Wr,
                                         const int32_t* topk_ids, const float* gates, const float* dgates,
                                         float* dWr, float* dbias, void* dx, void* ws, size_t ws_bytes,
                                         moeblaze_stream stream) {
  moeblaze_status r = check_router_shape(s);
  if (r != MOEBLAZE_OK) return r;
  if (!ok_ptr4(Wr) || !ok_ptr4(dWr) || (dbias && !ok_ptr4(dbias))) return MOEBLAZE_ERR_INVALID_ARG;
  if (s->L > 0 && (!ok_ptr(x) || !ok_ptr4(topk_ids) || !ok_ptr4(gates) || !ok_ptr4(dgates) || (dx && !ok_ptr(dx))))
    return MOEBLAZE_ERR_INVALID_ARG;
  if (ws_bytes < router_ws_bytes(*s)) return MOEBLAZE_ERR_WORKSPACE;
  if (s->L > 0 && !ok_ptr(ws)) return MOEBLAZE_ERR_INVALID_ARG;
  return launch_router_backward(*s, x, Wr, topk_ids, gates, dgates, dWr, dbias, dx, ws,
                                reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
