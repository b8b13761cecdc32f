// Gather + weighted combine of the identity expert (y[t] = sum_k g[t,k] x[t]
// through the index structures), the data movement of MoEBlaze's forward
// gather and fused write-back with the expert MLP taken out (MoEBlaze,
// awesome-system-papers page, section "免物化 token dispatch", Forward and
// Backward; the backward is the same kernel on dY -> dX).
//
// Schedule: one CTA per window of 8 tokens, all columns.  The window's
// 8*K (token, slot) positions are read from token_index_map and ranked
// ascending, which is expert-major order restricted to the window (the order
// the grouped expert GEMM walks its rows).  The CTA then walks them in that
// order, reading each routed row through expert_token_indices (the gather)
// and adding g * row into fp32 register accumulators, one chunk of 1024
// (bf16) or 512 (fp32) columns at a time with eight 16-byte row loads in
// flight per thread; every thread owns the same columns of all 8 rows, so the
// accumulation needs no atomics and the sorted list is built once per window.  Each output row is written once, each input row is read
// from HBM once (its K reads fall inside one CTA), the routed (L*K, d)
// buffer never exists.
#include <climits>

#include "common.cuh"

namespace moeblaze {
namespace {

constexpr int kWin = 8;        // tokens per CTA (the accumulator switch below has 8 rows)
constexpr int kThreads = 128;  // 16 bytes per thread per row

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(uint4 u, float* f) {
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  __device__ static void store(__nv_bfloat16* p, const float* f) {
    uint4 u;
    u.x = pack_bf16x2(f[0], f[1]); u.y = pack_bf16x2(f[2], f[3]);
    u.z = pack_bf16x2(f[4], f[5]); u.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4*>(p) = u;
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(uint4 u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ static void store(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreads) identity_combine_kernel(const T* __restrict__ src,
                                                                    const int32_t* __restrict__ D1,
                                                                    const int32_t* __restrict__ D4,
                                                                    const float* __restrict__ gates,
                                                                    T* __restrict__ dst, int64_t L, int d, int K,
                                                                    int64_t LK) {
  constexpr int V = Vec<T>::N;
  __shared__ int32_t pos_in[kWin * kMaxK], pos_s[kWin * kMaxK], tok_s[kWin * kMaxK];
  __shared__ float g_in[kWin * kMaxK], g_s[kWin * kMaxK];

  const int tid = threadIdx.x;
  const int64_t t0 = (int64_t)blockIdx.x * kWin;
  const int n = kWin * K;

  if (tid < n) {
    const int64_t t = t0 + tid / K;
    int32_t p = INT_MAX;
    float g = 0.f;
    if (t < L) {
      const int32_t q = D4[t * K + (tid % K)];
      if (q >= 0 && q < LK) { p = q; g = gates[t * K + (tid % K)]; }
    }
    pos_in[tid] = p;
    g_in[tid] = g;
  }
  __syncthreads();
  if (tid < n) {  // rank = place in ascending position order (expert-major)
    const int32_t p = pos_in[tid];
    int r = 0;
    for (int j = 0; j < n; ++j) r += (pos_in[j] < p) || (pos_in[j] == p && j < tid);
    pos_s[r] = p;
    g_s[r] = g_in[tid];
  }
  __syncthreads();
  if (tid < n) {  // the gather index; entries outside the window are dropped
    const int32_t tok = (pos_s[tid] != INT_MAX) ? D1[pos_s[tid]] : -1;
    tok_s[tid] = (tok >= 0 && tok - t0 >= 0 && tok - t0 < kWin) ? (int32_t)(tok - t0) : -1;
  }
  __syncthreads();

  // The same sorted list serves every column chunk of the window's rows.
  // Each thread keeps its columns of all 8 rows in registers; the row of an
  // entry is the same for every thread, so the switch below selects a
  // register accumulator without divergence.
  for (int cb = 0; cb < d; cb += kThreads * V) {
    const int col = cb + tid * V;
    if (col >= d) break;
    float acc[kWin][V];
#pragma unroll
    for (int j = 0; j < kWin; ++j)
#pragma unroll
      for (int c = 0; c < V; ++c) acc[j][c] = 0.f;
    constexpr int U = 8;
    for (int i0 = 0; i0 < n; i0 += U) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u;
        const int j = (i < n) ? tok_s[i] : -1;
        raw[u] = (j >= 0) ? __ldg(reinterpret_cast<const uint4*>(src + (t0 + j) * d + col)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u;
        const int j = (i < n) ? tok_s[i] : -1;
        const float g = (i < n) ? g_s[i] : 0.f;
        float v[V];
        Vec<T>::unpack(raw[u], v);
        switch (j) {
#define MB_ACC_ROW(J)                                    \
  case J:                                                \
    _Pragma("unroll") for (int c = 0; c < V; ++c) acc[J][c] += g * v[c]; \
    break;
          MB_ACC_ROW(0) MB_ACC_ROW(1) MB_ACC_ROW(2) MB_ACC_ROW(3)
          MB_ACC_ROW(4) MB_ACC_ROW(5) MB_ACC_ROW(6) MB_ACC_ROW(7)
#undef MB_ACC_ROW
          default:
            break;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kWin; ++j) {
      if (t0 + j < L) Vec<T>::store(dst + (t0 + j) * d + col, acc[j]);
    }
  }
}

}  // namespace

moeblaze_status launch_identity_combine(const moeblaze_shape& s, const void* src, const moeblaze_dispatch& disp,
                                        const float* gates, void* dst, cudaStream_t st) {
  if (s.L == 0) return MOEBLAZE_OK;
  const int64_t LK = s.L * s.K;
  dim3 grid((unsigned)((s.L + kWin - 1) / kWin), 1);
  if (s.dtype == MOEBLAZE_BF16) {
    identity_combine_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(src), disp.expert_token_indices, disp.token_index_map, gates,
        reinterpret_cast<__nv_bfloat16*>(dst), s.L, s.d, s.K, LK);
  } else {
    identity_combine_kernel<float><<<grid, kThreads, 0, st>>>(
        reinterpret_cast<const float*>(src), disp.expert_token_indices, disp.token_index_map, gates,
        reinterpret_cast<float*>(dst), s.L, s.d, s.K, LK);
  }
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

}  // namespace moeblaze
