// Gather + weighted combine of the identity expert (y[t] = sum_k g[t,k] x[t]
// through the index structures), the data movement of MoEBlaze's forward
// gather and fused write-back with the expert MLP taken out (MoEBlaze,
// awesome-system-papers page, section "免物化 token dispatch", Forward and
// Backward; the backward is the same kernel on dY -> dX).
//
// Schedule: one CTA per window of 8 tokens, all columns.  The window's
// 8*K (token, slot) positions are read from token_index_map and ranked
// ascending, which is expert-major order restricted to the window (the order
// the grouped expert GEMM walks its rows).  Like the GEMM path's producer,
// the CTA then gathers those routed rows, through expert_token_indices and in
// that order, into a shared-memory tile with 16-byte cp.async (one 1 KB
// column chunk of every routed row per stage, two stages in flight); like its
// epilogue, it then combines: every output piece sums the staged slots of its
// row times their gates in registers and is written once.  No atomics; each
// source row is read from HBM once (its K slots fall in one CTA).  Each output row is written once, each input row is read
// from HBM once (its K reads fall inside one CTA), the routed (L*K, d)
// buffer never exists.
#include <climits>

#include "common.cuh"

namespace moeblaze {
namespace {

constexpr int kWin = 8;           // tokens per CTA
constexpr int kThreads = 256;
constexpr int kChunkBytes = 1024;  // bytes of one routed row per column chunk
constexpr int kStages = 2;         // column chunks in flight per CTA
constexpr int kPieces = kChunkBytes / 16;

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kThreads) identity_combine_kernel(const T* __restrict__ src,
                                                                    const int32_t* __restrict__ D1,
                                                                    const int32_t* __restrict__ D4,
                                                                    const float* __restrict__ gates,
                                                                    T* __restrict__ dst, int64_t L, int d, int K,
                                                                    int64_t LK, const int32_t* __restrict__ hdr,
                                                                    int E, int32_t* err) {
  constexpr int V = Vec<T>::N;                 // elements per 16-byte piece
  constexpr int CH = kChunkBytes / sizeof(T);  // columns per chunk
  extern __shared__ __align__(16) uint8_t stage[];  // [kStages][n][kChunkBytes]
  __shared__ int32_t pos_in[kWin * kMaxK], pos_s[kWin * kMaxK], tok_s[kWin * kMaxK];
  __shared__ float g_in[kWin * kMaxK], g_s[kWin * kMaxK];
  __shared__ int32_t slot_of[kWin][kMaxK];
  __shared__ float gate_of[kWin][kMaxK];
  __shared__ int32_t nslot[kWin];

  const int tid = threadIdx.x;
  const int64_t t0 = (int64_t)blockIdx.x * kWin;
  const int n = kWin * K;
  // a dispatch built for another (L, E, K): record it and read none of its maps
  if (!meta_matches(hdr, L, E, K)) {
    if (tid == 0) atomicOr(err, kErrShapeMismatch);
    return;
  }

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
  if (tid < kWin) {  // the staged slots (expert-major) that belong to window row tid
    int m = 0;
    for (int i = 0; i < n; ++i)
      if (tok_s[i] == tid && m < kMaxK) { slot_of[tid][m] = i; gate_of[tid][m] = g_s[i]; ++m; }
    nslot[tid] = m;
  }
  __syncthreads();

  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
  const int nchunks = (d + CH - 1) / CH;
  // gather: the n routed rows of chunk c, in expert-major order, into buffer c % kStages
  auto gather = [&](int c) {
    const int col0 = c * CH;
    const uint32_t buf = sbase + (c % kStages) * n * kChunkBytes;
    for (int pc = tid; pc < n * kPieces; pc += kThreads) {
      const int i = pc / kPieces, off = pc % kPieces;
      const int j = tok_s[i];
      const int col = col0 + off * V;
      if (j >= 0 && col < d) cp_async16(buf + i * kChunkBytes + off * 16, src + (t0 + j) * d + col);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // combine: each output piece sums its row's staged slots with their gates
  auto combine = [&](int c) {
    const int col0 = c * CH;
    const uint8_t* buf = stage + (c % kStages) * n * kChunkBytes;
    for (int pc = tid; pc < kWin * kPieces; pc += kThreads) {
      const int j = pc / kPieces, off = pc % kPieces;
      const int col = col0 + off * V;
      if (t0 + j >= L || col >= d) continue;
      float acc[V];
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = 0.f;
      for (int m = 0; m < nslot[j]; ++m) {
        float v[V];
        Vec<T>::unpack(*reinterpret_cast<const uint4*>(buf + slot_of[j][m] * kChunkBytes + off * 16), v);
        const float g = gate_of[j][m];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] += g * v[e];
      }
      Vec<T>::store(dst + (t0 + j) * d + col, acc);
    }
  };
  // kStages chunks in flight while chunk c is awaited; one commit group per
  // chunk (empty past the end)
#pragma unroll
  for (int c = 0; c < kStages - 1; ++c) {
    if (c < nchunks) gather(c);
    else asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int c = 0; c < nchunks; ++c) {
    // chunk c + kStages - 1 goes into the buffer chunk c - 1 used (combined
    // before the trailing barrier of the previous iteration)
    if (c + kStages - 1 < nchunks) gather(c + kStages - 1);
    else asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
    __syncthreads();  // chunk c landed for every thread
    combine(c);
    __syncthreads();  // chunk c's buffer may be refilled
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Gate gradients of the identity expert: dg[t,k] = <dY[t], x[t]> for every
// slot k (the expert's output is the token itself).  One warp per token.
template <typename T>
__global__ void __launch_bounds__(256) identity_dgates_kernel(const T* __restrict__ x, const T* __restrict__ dY,
                                                              float* __restrict__ dg, int64_t L, int d, int K) {
  constexpr int V = Vec<T>::N;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= L) return;
  float acc = 0.f;
  for (int c = lane * V; c < d; c += 32 * V) {
    float a[V], b[V];
    Vec<T>::unpack(__ldg(reinterpret_cast<const uint4*>(x + t * d + c)), a);
    Vec<T>::unpack(__ldg(reinterpret_cast<const uint4*>(dY + t * d + c)), b);
#pragma unroll
    for (int e = 0; e < V; ++e) acc += a[e] * b[e];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane < K) dg[t * K + lane] = acc;
}

}  // namespace

moeblaze_status launch_identity_dgates(const moeblaze_shape& s, const void* x, const void* dY, float* dgates,
                                       cudaStream_t st) {
  if (s.L == 0) return MOEBLAZE_OK;
  const unsigned grid = (unsigned)((s.L + 7) / 8);
  if (s.dtype == MOEBLAZE_BF16)
    identity_dgates_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x),
                                                                reinterpret_cast<const __nv_bfloat16*>(dY), dgates,
                                                                s.L, s.d, s.K);
  else
    identity_dgates_kernel<float><<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(x),
                                                        reinterpret_cast<const float*>(dY), dgates, s.L, s.d, s.K);
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

moeblaze_status launch_identity_combine(const moeblaze_shape& s, const void* src, const moeblaze_dispatch& disp,
                                        const float* gates, void* dst, cudaStream_t st) {
  if (s.L == 0) return MOEBLAZE_OK;
  const int64_t LK = s.L * s.K;
  const MetaView meta = meta_view(disp.meta, s.E);
  const dim3 grid((unsigned)((s.L + kWin - 1) / kWin));
  const size_t smem = kStages * (size_t)kWin * s.K * kChunkBytes;
  if (s.dtype == MOEBLAZE_BF16) {
    auto k = identity_combine_kernel<__nv_bfloat16>;
    MB_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    k<<<grid, kThreads, smem, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), disp.expert_token_indices,
                                    disp.token_index_map, gates, reinterpret_cast<__nv_bfloat16*>(dst), s.L, s.d,
                                    s.K, LK, meta.hdr, s.E, meta.err);
  } else {
    auto k = identity_combine_kernel<float>;
    MB_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    k<<<grid, kThreads, smem, st>>>(reinterpret_cast<const float*>(src), disp.expert_token_indices,
                                    disp.token_index_map, gates, reinterpret_cast<float*>(dst), s.L, s.d, s.K, LK,
                                    meta.hdr, s.E, meta.err);
  }
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

}  // namespace moeblaze
