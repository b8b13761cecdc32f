// Internal declarations of the moeblaze library: shape-derived sizes, the
// layout of the dispatch meta buffer, inline-PTX wrappers for mbarrier, TMA
// and tcgen05 (sm_103a), and the launchers each .cu file provides.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moeblaze.h"

namespace moeblaze {

// ---------------------------------------------------------------- constants
constexpr int kChunkTokens = 1024;       // tokens per dispatch chunk (32 bitmap words)
constexpr int kChunkWords = kChunkTokens / 32;
constexpr int kRowPad = 256;             // expert row segments are padded to this (a pair of GEMM M tiles)
constexpr int kTileM = 128;              // rows of one GEMM tile
constexpr int kMaxE = 512;
constexpr int kMaxK = 8;
constexpr size_t kSchedBytes = 256;  // tile counters behind the fp32 accumulator of a bf16 forward/backward

// device error word bits
constexpr int kErrBadRouting = 1;
constexpr int kErrTimeout = 2;
constexpr int kErrShapeMismatch = 4;  // forward/backward given a dispatch built for another L, E or K

// ---------------------------------------------------------------- meta layout
// The meta buffer written by the dispatch build and read by the GEMMs:
//   int32 header[8]          err, num_m_tiles, padded_rows, L, E, K, reserved...
//   int32 n_e[E]             tokens per expert
//   int32 pad_off[E+1]       padded row offset of each expert (multiples of 256)
//   int32 order[E]           experts by descending n_e (ties: lower id first)
//   int32 tile_expert[MT]    expert of each 128-row tile, MT = max_m_tiles (an even count per expert)
constexpr int kHdrL = 3, kHdrE = 4, kHdrK = 5;  // header words holding the shape the build was made for
struct MetaView {
  int32_t* hdr;
  int32_t* err;
  int32_t* num_m_tiles;
  int32_t* padded_rows;
  int32_t* n_e;
  int32_t* pad_off;
  int32_t* order;
  int32_t* tile_expert;
};

inline int64_t max_padded_rows(int64_t LK, int E) {
  int64_t r = LK + (int64_t)E * (kRowPad - 1);
  return (r + kRowPad - 1) / kRowPad * kRowPad;
}
inline int64_t max_m_tiles(int64_t LK, int E) { return max_padded_rows(LK, E) / kTileM; }
inline int64_t num_chunks(int64_t L) { return (L + kChunkTokens - 1) / kChunkTokens; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline MetaView meta_view(void* meta, int E) {
  int32_t* p = reinterpret_cast<int32_t*>(meta);
  MetaView m;
  m.hdr = p;
  m.err = p + 0;
  m.num_m_tiles = p + 1;
  m.padded_rows = p + 2;
  int32_t* q = p + 8;
  m.n_e = q; q += E;
  m.pad_off = q; q += E + 1;
  m.order = q; q += E;
  m.tile_expert = q;
  return m;
}
inline size_t meta_bytes(int64_t LK, int E) {
  return align_up(sizeof(int32_t) * (8 + E + (E + 1) + E + (size_t)max_m_tiles(LK, E)), 256);
}

// The shape a dispatch build recorded in its meta header against the shape a
// forward/backward call was given.  The tile table, offsets and counts are
// sized and laid out by (L, E, K), so a kernel reads nothing else of the
// dispatch unless this holds.  Used by the kernels on the device header and
// by moeblaze_dispatch_meta_check on a host copy of it.  A build for L = 0
// records only L (no kernel reads its structures).
__host__ __device__ inline bool meta_matches(const int32_t* hdr, int64_t L, int E, int K) {
  return (int64_t)hdr[kHdrL] == L && (L == 0 || (hdr[kHdrE] == E && hdr[kHdrK] == K));
}

// ---------------------------------------------------------------- status helper
#define MB_CUDA(call)                                           \
  do {                                                          \
    cudaError_t e_ = (call);                                    \
    if (e_ != cudaSuccess) return MOEBLAZE_ERR_CUDA;            \
  } while (0)

// ---------------------------------------------------------------- launchers
// dispatch.cu
moeblaze_status launch_dispatch(const moeblaze_shape& s, const int32_t* ids, const moeblaze_dispatch& out,
                                void* ws, cudaStream_t st);
size_t dispatch_ws_bytes(const moeblaze_shape& s);
// the dispatch build on the library's fixed scratch array (see dispatch.cu)
moeblaze_status launch_dispatch_static(const moeblaze_shape& s, const int32_t* ids, const moeblaze_dispatch& out,
                                       cudaStream_t st);
// the dispatch scratch's packed (in-chunk rank << 16 | expert) slots [L][K]
// and per-(expert, chunk) counts [E][C], for a kernel that does K1's work
void dispatch_ws_parts(const moeblaze_shape& s, void* ws, int32_t** packed, int32_t** cnt);
// K2 (large layers) and K3 on a scratch whose slots and counts are written
moeblaze_status launch_dispatch_tail(const moeblaze_shape& s, const moeblaze_dispatch& out, void* ws, cudaStream_t st);

// identity.cu
moeblaze_status launch_identity_combine(const moeblaze_shape& s, const void* src, const moeblaze_dispatch& disp,
                                        const float* gates, void* dst, cudaStream_t st);
moeblaze_status launch_identity_dgates(const moeblaze_shape& s, const void* x, const void* dY, float* dgates,
                                       cudaStream_t st);

// simt.cu (fp32 path)
moeblaze_status simt_forward(const moeblaze_shape& s, const float* x, const float* gates,
                             const moeblaze_dispatch& disp, const float* W1, const float* W2, const float* W3,
                             float* y, float* saved, float* wsH, cudaStream_t st);
moeblaze_status simt_backward(const moeblaze_shape& s, const float* dY, const float* x, const float* gates,
                              const moeblaze_dispatch& disp, const float* W1, const float* W2, const float* W3,
                              const float* saved, float* dX, float* dW1, float* dW2, float* dW3, float* dgates,
                              float* wsdAB, float* wsHg, cudaStream_t st);

// gemm_tc.cu (bf16 tensor-core path).  wsH / wsHg NULL selects the
// recompute variants (MOEBLAZE_RECOMPUTE_H), which keep the row gates in
// `saved`; the backward overwrites the saved A, B with dA, dB.
moeblaze_status tc_forward(const moeblaze_shape& s, const __nv_bfloat16* x, const float* gates,
                           const moeblaze_dispatch& disp, const __nv_bfloat16* W1, const __nv_bfloat16* W2,
                           const __nv_bfloat16* W3, __nv_bfloat16* y, __nv_bfloat16* saved, __nv_bfloat16* wsH,
                           float* wsY32, cudaStream_t st);
moeblaze_status tc_backward(const moeblaze_shape& s, const __nv_bfloat16* dY, const __nv_bfloat16* x,
                            const float* gates, const moeblaze_dispatch& disp, const __nv_bfloat16* W1,
                            const __nv_bfloat16* W2, const __nv_bfloat16* W3, __nv_bfloat16* saved,
                            __nv_bfloat16* dX, __nv_bfloat16* dW1, __nv_bfloat16* dW2, __nv_bfloat16* dW3,
                            float* dgates, __nv_bfloat16* wsHg, float* wsdX32, cudaStream_t st);

// router.cu
constexpr int kMaxRouterE = 256;
size_t router_ws_bytes(const moeblaze_shape& s);
moeblaze_status launch_router_forward(const moeblaze_shape& s, const void* x, const float* Wr, const float* bias,
                                      int32_t* ids, float* gates, cudaStream_t st);
moeblaze_status launch_router_backward(const moeblaze_shape& s, const void* x, const float* Wr, const int32_t* ids,
                                       const float* gates, const float* dgates, float* dWr, float* dbias, void* dx,
                                       void* ws, cudaStream_t st);

// router_tc.cu: the router fused with the dispatch's first step (bf16 x, E <= 64)
bool router_dispatch_fused(const moeblaze_shape& s);
size_t router_dispatch_ws_bytes(const moeblaze_shape& s);
moeblaze_status launch_router_dispatch(const moeblaze_shape& s, const void* x, const float* Wr, const float* bias,
                                       int32_t* ids, float* gates, const moeblaze_dispatch& out, void* ws,
                                       cudaStream_t st);

// shared helpers (abi.cu)
int sm_count();
void count_launch(int n = 1);
// record stage-boundary event i on st if the caller asked for it
void stage_event(int i, cudaStream_t st);
// the calling thread's failure-path test settings (moeblaze_set_fault_injection):
// wait limit in ns (0: the default) and whether the down projection withholds a stage
void fault_injection(uint64_t* wait_ns, int* withhold);

// ---------------------------------------------------------------- device helpers

// bf16x2 packing of two fp32 values, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace moeblaze
