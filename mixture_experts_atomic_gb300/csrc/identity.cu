// Gather + weighted combine of the identity expert (y[t] = sum_k g[t,k] x[t]
// through the index structures), the data movement of MoEBlaze's forward
// gather and fused write-back with the expert MLP taken out (MoEBlaze,
// awesome-system-papers page, section "免物化 token dispatch", Forward and
// Backward; the backward is the same kernel on dY -> dX).
//
// Schedule: one CTA per window of 8 tokens, all columns.  The window's 8*K
// (token, slot) positions are read from token_index_map and ranked
// ascending, which is expert-major order restricted to the window (the order
// the grouped expert GEMM walks its rows).  Like the GEMM path's producer,
// the CTA then gathers those routed rows, through expert_token_indices and in
// that order, into a shared-memory tile with 16-byte cp.async (one 256-byte
// column chunk of every routed row per stage, two stages in flight); like its
// epilogue, it then combines: every output piece sums the staged slots of its
// row times their gates (packed fp32x2 FMAs, fp32 accumulation) and is
// written once.  A thread copies and combines the same 16-byte column piece
// of its rows in every chunk, so its source, shared-memory and output
// addresses are computed once per window.  No atomics; each output row is
// written once; the K routed rows of a token fall inside one CTA, so HBM
// serves each source row once and L2 the repeats; the routed (L*K, d) buffer
// never exists.  Small CTAs (four warps, 16 KB of stages for K = 4) keep
// many windows resident per SM, so the latency of one window's chunk barrier
// hides behind the others (measured on the 2M-token, 256-expert layer:
// 1 KB chunks and 256 threads 12.7 ms a pass, 256 B and 128 threads 9.8 ms).
#include <climits>

#include "common.cuh"

namespace moeblaze {
namespace {

constexpr int kWin = 8;            // tokens per CTA
constexpr int kThreads = 128;
constexpr int kChunkBytes = 256;   // bytes of one routed row per column chunk
constexpr int kStages = 2;         // column chunks in flight per CTA
constexpr int kPieces = kChunkBytes / 16;        // 16-byte pieces of a row chunk
constexpr int kRowsPerPass = kThreads / kPieces;  // rows the block covers per pass (8)

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(uint4 u, float* f) {
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  // acc[i] += g * (elements 2i, 2i+1 of the 16-byte piece u)
  __device__ static void fma(uint4 u, float2 g, float2* acc) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)  // bf16 -> fp32 is exact: the 16 bits become the high half
      acc[i] = __ffma2_rn(make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u)), g, acc[i]);
  }
  __device__ static uint4 pack(const float2* acc) {
    return make_uint4(pack_bf16x2(acc[0].x, acc[0].y), pack_bf16x2(acc[1].x, acc[1].y),
                      pack_bf16x2(acc[2].x, acc[2].y), pack_bf16x2(acc[3].x, acc[3].y));
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(uint4 u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ static void fma(uint4 u, float2 g, float2* acc) {
    acc[0] = __ffma2_rn(make_float2(__uint_as_float(u.x), __uint_as_float(u.y)), g, acc[0]);
    acc[1] = __ffma2_rn(make_float2(__uint_as_float(u.z), __uint_as_float(u.w)), g, acc[1]);
  }
  __device__ static uint4 pack(const float2* acc) {
    return make_uint4(__float_as_uint(acc[0].x), __float_as_uint(acc[0].y), __float_as_uint(acc[1].x),
                      __float_as_uint(acc[1].y));
  }
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// KM: the largest K this instance handles (4 or kMaxK), which sizes the
// per-thread address tables held in registers.
template <typename T, int KM>
__global__ void __launch_bounds__(kThreads) identity_combine_kernel(const T* __restrict__ src,
                                                                    const int32_t* __restrict__ D1,
                                                                    const int32_t* __restrict__ D4,
                                                                    const float* __restrict__ gates,
                                                                    T* __restrict__ dst, int64_t L, int d, int K,
                                                                    int64_t LK, const int32_t* __restrict__ hdr,
                                                                    int E, int32_t* err) {
  constexpr int V = Vec<T>::N;                 // elements per 16-byte piece
  constexpr int CH = kChunkBytes / sizeof(T);  // columns per chunk
  constexpr int kGatherIt = kWin * KM / kRowsPerPass;  // routed rows a thread copies (per chunk)
  constexpr int kCombineIt = kWin / kRowsPerPass;      // output rows a thread writes (per chunk)
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
    tok_s[tid] = (tok >= 0 && tok < L && tok - t0 >= 0 && tok - t0 < kWin) ? (int32_t)(tok - t0) : -1;
  }
  __syncthreads();
  if (tid < kWin) {  // the staged slots (expert-major) that belong to window row tid
    int m = 0;
    for (int i = 0; i < n; ++i)
      if (tok_s[i] == tid && m < kMaxK) { slot_of[tid][m] = i; gate_of[tid][m] = g_s[i]; ++m; }
    nslot[tid] = m;
  }
  __syncthreads();

  // This thread's 16-byte piece `off` of every row chunk, and the rows it
  // handles: routed rows r0, r0 + 4, ... (gather) and window rows r0, r0 + 4
  // (combine).  Their addresses are fixed for the whole window.
  const int off = tid % kPieces;
  const int r0 = tid / kPieces;
  const int dp = (int)(((int64_t)d * sizeof(T)) / 16);  // 16-byte pieces of a row
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
  const T* gsrc[kGatherIt];
#pragma unroll
  for (int it = 0; it < kGatherIt; ++it) {
    const int i = r0 + kRowsPerPass * it;
    gsrc[it] = (i < n && tok_s[i] >= 0) ? src + (t0 + tok_s[i]) * d + off * V : nullptr;
  }
  int ns[kCombineIt];
  uint32_t soff[kCombineIt][KM];
  float2 sg[kCombineIt][KM];
  T* ydst[kCombineIt];
#pragma unroll
  for (int it = 0; it < kCombineIt; ++it) {
    const int j = r0 + kRowsPerPass * it;
    ns[it] = (t0 + j < L) ? min(nslot[j], KM) : 0;
    ydst[it] = dst + (t0 + j) * d + off * V;
#pragma unroll
    for (int m = 0; m < KM; ++m) {
      soff[it][m] = (uint32_t)slot_of[j][m] * kChunkBytes + off * 16;
      sg[it][m] = make_float2(gate_of[j][m], gate_of[j][m]);
    }
  }
  const int nchunks = (d + CH - 1) / CH;
  // gather: this thread's pieces of the n routed rows of chunk c, in
  // expert-major row order, into buffer c % kStages
  auto gather = [&](int c) {
    const uint32_t buf = sbase + (uint32_t)((c % kStages) * n * kChunkBytes + r0 * kChunkBytes + off * 16);
    if (c * kPieces + off < dp) {
#pragma unroll
      for (int it = 0; it < kGatherIt; ++it)
        if (gsrc[it]) cp_async16(buf + it * kRowsPerPass * kChunkBytes, gsrc[it] + (int64_t)c * CH);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // combine: each output piece sums its row's staged slots with their gates
  auto combine = [&](int c) {
    if (c * kPieces + off >= dp) return;
    const uint8_t* buf = stage + (c % kStages) * n * kChunkBytes;
#pragma unroll
    for (int it = 0; it < kCombineIt; ++it) {
      if (ns[it] == 0) continue;
      float2 acc[V / 2];
#pragma unroll
      for (int i = 0; i < V / 2; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < KM; ++m)
        if (m < ns[it]) Vec<T>::fma(*reinterpret_cast<const uint4*>(buf + soff[it][m]), sg[it][m], acc);
      *reinterpret_cast<uint4*>(ydst[it] + (int64_t)c * CH) = Vec<T>::pack(acc);
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
  // one instance per element type and K range (the address tables are sized by the largest K)
  auto run = [&](auto kern, const auto* in, auto* out) -> moeblaze_status {
    MB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    kern<<<grid, kThreads, smem, st>>>(in, disp.expert_token_indices, disp.token_index_map, gates, out, s.L, s.d, s.K,
                                       LK, meta.hdr, s.E, meta.err);
    MB_CUDA(cudaGetLastError());
    return MOEBLAZE_OK;
  };
  moeblaze_status r;
  if (s.dtype == MOEBLAZE_BF16) {
    const auto* in = reinterpret_cast<const __nv_bfloat16*>(src);
    auto* out = reinterpret_cast<__nv_bfloat16*>(dst);
    r = s.K <= 4 ? run(identity_combine_kernel<__nv_bfloat16, 4>, in, out)
                 : run(identity_combine_kernel<__nv_bfloat16, kMaxK>, in, out);
  } else {
    const auto* in = reinterpret_cast<const float*>(src);
    auto* out = reinterpret_cast<float*>(dst);
    r = s.K <= 4 ? run(identity_combine_kernel<float, 4>, in, out) : run(identity_combine_kernel<float, kMaxK>, in, out);
  }
  if (r != MOEBLAZE_OK) return r;
  count_launch();
  return MOEBLAZE_OK;
}

}  // namespace moeblaze
