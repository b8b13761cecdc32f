// Token-choice top-K softmax router and its backward: the step before the
// dispatch of MoEBlaze (awesome-system-papers page, assumptions of the
// problem statement: token-choice, top-K routing over the L routed tokens).
//
//   logits[t,e] = x[t] . Wr[:,e] (+ bias[e])            fp32, Wr (d,E) fp32
//   ids[t,0..K) = the K largest logits, equal logits to the lower expert
//                 index, slot 0 the largest
//   gates[t,k]  = softmax over the K selected logits
//
// backward, given dgates (from moeblaze_backward):
//   dlogit[t, ids[t,k]] = g_k (dg_k - sum_j g_j dg_j)    (0 for the others)
//   dx = dlogit Wr^T,  dWr = x^T dlogit,  dbias = sum_t dlogit[t]
//
// Both directions are small GEMMs with N = E (at most 256) on CUDA cores in
// fp32: a CTA owns a 64-row tile and the fp32 products are register-blocked
// over the experts.  The weight-gradient sums are split over token ranges
// into per-split partials that a last kernel adds in a fixed order, so every
// result is bitwise repeatable.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace moeblaze {
namespace {

constexpr int kRT = 64;        // rows of a CTA tile (tokens, or rows of Wr)
constexpr int kRK = 32;        // reduction chunk staged in shared memory
constexpr int kRThreads = 256;

// thread layout of a 64 x EP tile: TE threads across the experts (expert
// e = j * TE + te for j < EPT), TTH threads across the rows (RPT rows each)
template <int EP>
struct RLayout {
  static constexpr int TE = EP <= 32 ? 8 : 16;
  static constexpr int EPT = EP / TE;
  static constexpr int TTH = kRThreads / TE;
  static constexpr int RPT = kRT / TTH;
};

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), e = unpack_bf16x2(u.w);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y; v[4] = c.x; v[5] = c.y; v[6] = e.x; v[7] = e.y;
}
__device__ __forceinline__ void load8(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                            pack_bf16x2(v[6], v[7]));
}
__device__ __forceinline__ void store8(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// acc[i][j] += sum_c A[row_i][c] * B[c][expert_j] over one staged chunk
template <int EP>
__device__ __forceinline__ void tile_fma(const float (*As)[kRK + 1], const float (*Bs)[EP], int te, int tr,
                                         float (&acc)[RLayout<EP>::RPT][RLayout<EP>::EPT]) {
  using Ly = RLayout<EP>;
#pragma unroll 4
  for (int c = 0; c < kRK; ++c) {
    float av[Ly::RPT], bv[Ly::EPT];
#pragma unroll
    for (int i = 0; i < Ly::RPT; ++i) av[i] = As[tr * Ly::RPT + i][c];
#pragma unroll
    for (int j = 0; j < Ly::EPT; ++j) bv[j] = Bs[c][j * Ly::TE + te];
#pragma unroll
    for (int i = 0; i < Ly::RPT; ++i)
#pragma unroll
      for (int j = 0; j < Ly::EPT; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
}

// ------------------------------------------------------------------ forward
template <typename T, int EP>
__global__ void __launch_bounds__(kRThreads) router_fwd_kernel(const T* __restrict__ x, const float* __restrict__ Wr,
                                                               const float* __restrict__ bias, int64_t L, int d, int E,
                                                               int K, int32_t* __restrict__ ids,
                                                               float* __restrict__ gates) {
  using Ly = RLayout<EP>;
  __shared__ float xs[kRT][kRK + 1];
  __shared__ __align__(16) float ws[kRK][EP];
  const int tid = threadIdx.x, te = tid % Ly::TE, tr = tid / Ly::TE;
  const int64_t t0 = (int64_t)blockIdx.x * kRT;
  float acc[Ly::RPT][Ly::EPT];
#pragma unroll
  for (int i = 0; i < Ly::RPT; ++i)
#pragma unroll
    for (int j = 0; j < Ly::EPT; ++j) acc[i][j] = 0.f;

  const int lr = tid >> 2, lc = (tid & 3) * 8;  // this thread's 8 elements of the 64 x 32 x tile
  for (int k0 = 0; k0 < d; k0 += kRK) {
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (t0 + lr < L) load8(x + (t0 + lr) * d + k0 + lc, v);
#pragma unroll
    for (int u = 0; u < 8; ++u) xs[lr][lc + u] = v[u];
    for (int i = tid; i < kRK * EP; i += kRThreads) {
      const int r = i / EP, c = i % EP;
      ws[r][c] = c < E ? Wr[(int64_t)(k0 + r) * E + c] : 0.f;
    }
    __syncthreads();
    tile_fma<EP>(xs, ws, te, tr, acc);
    __syncthreads();
  }

  // bias; the padding experts (e >= E) can never be chosen
#pragma unroll
  for (int j = 0; j < Ly::EPT; ++j) {
    const int e = j * Ly::TE + te;
    const float b = (e < E && bias) ? bias[e] : 0.f;
#pragma unroll
    for (int i = 0; i < Ly::RPT; ++i) acc[i][j] = e < E ? acc[i][j] + b : -FLT_MAX;
  }

  // top-K of each row across the TE lanes that hold its experts (consecutive
  // lanes of one warp): K rounds of a segmented arg-max, larger logit first,
  // equal logits to the lower index; the owner lane marks the winner taken
#pragma unroll
  for (int i = 0; i < Ly::RPT; ++i) {
    uint32_t taken = 0;
    float selv[kMaxK];
    int seli[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      selv[k] = 0.f;
      seli[k] = 0;
      if (k < K) {
        float bv = -FLT_MAX;
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < Ly::EPT; ++j) {
          const int e = j * Ly::TE + te;
          const float a = acc[i][j];
          if (!((taken >> j) & 1u) && e < E && (a > bv || (a == bv && e < bi))) {
            bv = a;
            bi = e;
          }
        }
#pragma unroll
        for (int off = Ly::TE / 2; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        selv[k] = bv;
        seli[k] = bi;
        if (bi % Ly::TE == te) taken |= 1u << (bi / Ly::TE);
      }
    }
    const int64_t t = t0 + tr * Ly::RPT + i;
    if (te == 0 && t < L) {
      float w[kMaxK], sum = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        w[k] = k < K ? expf(selv[k] - selv[0]) : 0.f;
        sum += w[k];
      }
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        if (k < K) {
          ids[t * K + k] = seli[k];
          gates[t * K + k] = w[k] / sum;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ backward
// dlogit of the selected experts (kept in the workspace for dWr) and
// dx = dlogit Wr^T for one 64-token tile
template <typename T, int EP>
__global__ void __launch_bounds__(kRThreads) router_dx_kernel(const float* __restrict__ Wr,
                                                              const int32_t* __restrict__ ids,
                                                              const float* __restrict__ gates,
                                                              const float* __restrict__ dgates, int64_t L, int d, int E,
                                                              int K, float* __restrict__ dl, T* __restrict__ dx) {
  __shared__ float dls[kRT][kMaxK];
  __shared__ int ids_s[kRT][kMaxK];
  __shared__ float ws[kRK][EP + 1];
  const int tid = threadIdx.x;
  const int64_t t0 = (int64_t)blockIdx.x * kRT;
  if (tid < kRT) {
    const int64_t t = t0 + tid;
    float g[kMaxK], dg[kMaxK], s = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      g[k] = (k < K && t < L) ? gates[t * K + k] : 0.f;
      dg[k] = (k < K && t < L) ? dgates[t * K + k] : 0.f;
      ids_s[tid][k] = (k < K && t < L) ? ids[t * K + k] : 0;
      s = fmaf(g[k], dg[k], s);
    }
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      const float v = g[k] * (dg[k] - s);
      dls[tid][k] = k < K ? v : 0.f;
      if (k < K && t < L) dl[t * K + k] = v;
    }
  }
  __syncthreads();
  if (!dx) return;
  const int row = tid >> 2, c8 = (tid & 3) * 8;
  for (int k0 = 0; k0 < d; k0 += kRK) {
    for (int i = tid; i < kRK * EP; i += kRThreads) {
      const int r = i / EP, c = i % EP;
      ws[r][c] = c < E ? Wr[(int64_t)(k0 + r) * E + c] : 0.f;
    }
    __syncthreads();
    float out[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float a = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxK; ++k)
        if (k < K && (unsigned)ids_s[row][k] < (unsigned)E) a = fmaf(dls[row][k], ws[c8 + u][ids_s[row][k]], a);
      out[u] = a;
    }
    if (t0 + row < L) store8(dx + (t0 + row) * d + k0 + c8, out);
    __syncthreads();
  }
}

// partial dWr (and dbias) of one 64-row block of Wr over one token split:
// part[s][j][e] = sum_{t in split s} x[t, j] dlogit[t, e]
template <typename T, int EP>
__global__ void __launch_bounds__(kRThreads) router_dwr_kernel(const T* __restrict__ x, const int32_t* __restrict__ ids,
                                                               const float* __restrict__ dl, int64_t L, int d, int E,
                                                               int K, int64_t split, float* __restrict__ part,
                                                               float* __restrict__ part_b) {
  using Ly = RLayout<EP>;
  __shared__ float xs[kRT][kRK + 1];            // xs[j][c] = x[t_c, j0 + j]
  __shared__ __align__(16) float ds[kRK][EP];   // ds[c][e] = dlogit[t_c, e]
  const int tid = threadIdx.x, te = tid % Ly::TE, tr = tid / Ly::TE;
  const int j0 = blockIdx.x * kRT;
  const int64_t ts = (int64_t)blockIdx.y * split;
  const int64_t tend = min(L, ts + split);
  float acc[Ly::RPT][Ly::EPT];
#pragma unroll
  for (int i = 0; i < Ly::RPT; ++i)
#pragma unroll
    for (int j = 0; j < Ly::EPT; ++j) acc[i][j] = 0.f;
  float bacc = 0.f;
  const int lc = tid >> 3, lj = (tid & 7) * 8;  // token lc of the chunk, columns lj..lj+7
  for (int64_t c0 = ts; c0 < tend; c0 += kRK) {
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (c0 + lc < tend) load8(x + (c0 + lc) * d + j0 + lj, v);
#pragma unroll
    for (int u = 0; u < 8; ++u) xs[lj + u][lc] = v[u];
    for (int i = tid; i < kRK * EP; i += kRThreads) (&ds[0][0])[i] = 0.f;
    __syncthreads();
    if (tid < kRK && c0 + tid < tend) {
      const int64_t t = c0 + tid;
      for (int k = 0; k < K; ++k) {
        const int e = ids[t * K + k];
        if ((unsigned)e < (unsigned)E) ds[tid][e] = dl[t * K + k];
      }
    }
    __syncthreads();
    tile_fma<EP>(xs, ds, te, tr, acc);
    if (blockIdx.x == 0 && tid < EP) {
      for (int c = 0; c < kRK; ++c) bacc += ds[c][tid];
    }
    __syncthreads();
  }
  float* dst = part + (int64_t)blockIdx.y * d * E;
#pragma unroll
  for (int i = 0; i < Ly::RPT; ++i) {
    const int j = j0 + tr * Ly::RPT + i;
#pragma unroll
    for (int jj = 0; jj < Ly::EPT; ++jj) {
      const int e = jj * Ly::TE + te;
      if (e < E) dst[(int64_t)j * E + e] = acc[i][jj];
    }
  }
  if (blockIdx.x == 0 && tid < E) part_b[(int64_t)blockIdx.y * E + tid] = bacc;
}

__global__ void router_reduce_kernel(const float* __restrict__ part, const float* __restrict__ part_b, int64_t n,
                                     int E, int S, float* __restrict__ dWr, float* __restrict__ dbias) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n + E; i += (int64_t)gridDim.x * blockDim.x) {
    if (i < n) {
      float a = 0.f;
      for (int s = 0; s < S; ++s) a += part[(int64_t)s * n + i];
      dWr[i] = a;
    } else if (dbias) {
      const int e = (int)(i - n);
      float a = 0.f;
      for (int s = 0; s < S; ++s) a += part_b[(int64_t)s * E + e];
      dbias[e] = a;
    }
  }
}

int padded_experts(int E) {
  int ep = 8;
  while (ep < E) ep *= 2;
  return ep;
}

// token splits of the weight-gradient sums: enough CTAs to fill the GPU a
// few times over, at least one 32-token chunk per split
int64_t router_splits(const moeblaze_shape& s) {
  const int64_t jb = s.d / kRT;
  int64_t S = (4 * (int64_t)sm_count() + jb - 1) / jb;
  const int64_t chunks = (s.L + kRK - 1) / kRK;
  if (S > chunks) S = chunks;
  return S < 1 ? 1 : S;
}

template <typename T, int EP>
moeblaze_status fwd_ep(const moeblaze_shape& s, const void* x, const float* Wr, const float* bias, int32_t* ids,
                       float* gates, cudaStream_t st) {
  const unsigned grid = (unsigned)((s.L + kRT - 1) / kRT);
  router_fwd_kernel<T, EP><<<grid, kRThreads, 0, st>>>(static_cast<const T*>(x), Wr, bias, s.L, s.d, s.E, s.K, ids,
                                                      gates);
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

template <typename T, int EP>
moeblaze_status bwd_ep(const moeblaze_shape& s, const void* x, const float* Wr, const int32_t* ids,
                       const float* gates, const float* dgates, float* dWr, float* dbias, void* dx, void* ws,
                       cudaStream_t st) {
  const int64_t S = router_splits(s);
  const int64_t split = ((s.L + S - 1) / S + kRK - 1) / kRK * kRK;
  char* w = static_cast<char*>(ws);
  float* dl = reinterpret_cast<float*>(w);
  float* part = reinterpret_cast<float*>(w + align_up(sizeof(float) * s.L * s.K, 256));
  float* part_b = part + (size_t)S * s.d * s.E;
  const unsigned tiles = (unsigned)((s.L + kRT - 1) / kRT);
  router_dx_kernel<T, EP><<<tiles, kRThreads, 0, st>>>(Wr, ids, gates, dgates, s.L, s.d, s.E, s.K, dl,
                                                       static_cast<T*>(dx));
  MB_CUDA(cudaGetLastError());
  router_dwr_kernel<T, EP><<<dim3((unsigned)(s.d / kRT), (unsigned)S), kRThreads, 0, st>>>(
      static_cast<const T*>(x), ids, dl, s.L, s.d, s.E, s.K, split, part, part_b);
  MB_CUDA(cudaGetLastError());
  const int64_t n = (int64_t)s.d * s.E;
  int64_t blocks = (n + s.E + 255) / 256;
  if (blocks > 8 * (int64_t)sm_count()) blocks = 8 * (int64_t)sm_count();
  router_reduce_kernel<<<(unsigned)blocks, 256, 0, st>>>(part, part_b, n, s.E, (int)S, dWr, dbias);
  MB_CUDA(cudaGetLastError());
  count_launch(3);
  return MOEBLAZE_OK;
}

template <typename T>
moeblaze_status fwd_t(const moeblaze_shape& s, const void* x, const float* Wr, const float* bias, int32_t* ids,
                      float* gates, cudaStream_t st) {
  switch (padded_experts(s.E)) {
    case 8: return fwd_ep<T, 8>(s, x, Wr, bias, ids, gates, st);
    case 16: return fwd_ep<T, 16>(s, x, Wr, bias, ids, gates, st);
    case 32: return fwd_ep<T, 32>(s, x, Wr, bias, ids, gates, st);
    case 64: return fwd_ep<T, 64>(s, x, Wr, bias, ids, gates, st);
    case 128: return fwd_ep<T, 128>(s, x, Wr, bias, ids, gates, st);
    case 256: return fwd_ep<T, 256>(s, x, Wr, bias, ids, gates, st);
  }
  return MOEBLAZE_ERR_UNSUPPORTED;
}

template <typename T>
moeblaze_status bwd_t(const moeblaze_shape& s, const void* x, const float* Wr, const int32_t* ids,
                      const float* gates, const float* dgates, float* dWr, float* dbias, void* dx, void* ws,
                      cudaStream_t st) {
  switch (padded_experts(s.E)) {
    case 8: return bwd_ep<T, 8>(s, x, Wr, ids, gates, dgates, dWr, dbias, dx, ws, st);
    case 16: return bwd_ep<T, 16>(s, x, Wr, ids, gates, dgates, dWr, dbias, dx, ws, st);
    case 32: return bwd_ep<T, 32>(s, x, Wr, ids, gates, dgates, dWr, dbias, dx, ws, st);
    case 64: return bwd_ep<T, 64>(s, x, Wr, ids, gates, dgates, dWr, dbias, dx, ws, st);
    case 128: return bwd_ep<T, 128>(s, x, Wr, ids, gates, dgates, dWr, dbias, dx, ws, st);
    case 256: return bwd_ep<T, 256>(s, x, Wr, ids, gates, dgates, dWr, dbias, dx, ws, st);
  }
  return MOEBLAZE_ERR_UNSUPPORTED;
}

}  // namespace

size_t router_ws_bytes(const moeblaze_shape& s) {
  const int64_t S = router_splits(s);
  return align_up(sizeof(float) * s.L * s.K, 256) + align_up(sizeof(float) * ((size_t)S * s.d * s.E + S * s.E), 256);
}

moeblaze_status launch_router_forward(const moeblaze_shape& s, const void* x, const float* Wr, const float* bias,
                                      int32_t* ids, float* gates, cudaStream_t st) {
  if (s.L == 0) return MOEBLAZE_OK;
  return s.dtype == MOEBLAZE_BF16 ? fwd_t<__nv_bfloat16>(s, x, Wr, bias, ids, gates, st)
                                  : fwd_t<float>(s, x, Wr, bias, ids, gates, st);
}

moeblaze_status launch_router_backward(const moeblaze_shape& s, const void* x, const float* Wr, const int32_t* ids,
                                       const float* gates, const float* dgates, float* dWr, float* dbias, void* dx,
                                       void* ws, cudaStream_t st) {
  if (s.L == 0) {
    MB_CUDA(cudaMemsetAsync(dWr, 0, sizeof(float) * s.d * s.E, st));
    if (dbias) MB_CUDA(cudaMemsetAsync(dbias, 0, sizeof(float) * s.E, st));
    return MOEBLAZE_OK;
  }
  return s.dtype == MOEBLAZE_BF16 ? bwd_t<__nv_bfloat16>(s, x, Wr, ids, gates, dgates, dWr, dbias, dx, ws, st)
                                  : bwd_t<float>(s, x, Wr, ids, gates, dgates, dWr, dbias, dx, ws, st);
}

}  // namespace moeblaze
