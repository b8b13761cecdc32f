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
// All three are small GEMMs with N = E (at most 256) on CUDA cores in fp32.
// A CTA owns a 64-row tile (tokens, or rows of Wr), its products are
// register-blocked over the experts, and the streamed operand (x, Wr) comes
// through a multi-stage cp.async pipeline of 64-wide chunks so that several
// chunks of every CTA are in flight.  The weight-gradient sums are split
// over token ranges into per-split partials that a last kernel adds in a
// fixed order, so every result is bitwise repeatable.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace moeblaze {
namespace {

constexpr int kRT = 64;        // rows of a CTA tile (tokens, or rows of Wr)
constexpr int kRC = 64;        // width of a streamed chunk
constexpr int kRThreads = 256;

// thread layout of a 64 x EP tile: TE threads across the experts (expert
// e = j * TE + te for j < EPT), TTH threads across the rows (RPT rows each)
template <int EP>
struct RLayout {
  static constexpr int TE = EP <= 32 ? 8 : 16;
  static constexpr int EPT = EP / TE;
  static constexpr int TTH = kRThreads / TE;
  static constexpr int RPT = kRT / TTH;
  static constexpr int STAGES = EP >= 128 ? 2 : 3;
};

// row pitch (elements) of a staged 64-wide chunk of x: 16-byte multiple, and
// rows 2 or 4 apart land on different banks
template <typename T>
struct XPitch {
  static constexpr int value = sizeof(T) == 2 ? 72 : 68;
};

__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

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

__device__ __forceinline__ void cp16(uint32_t dst, const void* src, bool valid) {
  // a 16-byte copy, zero-filled when !valid (the source is not read)
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// 64 rows x 64 columns of a row-major (rows, ld) matrix, rows >= nrows zero
template <typename T>
__device__ __forceinline__ void stage_rows(T* dst, const T* src, int64_t row0, int64_t nrows, int64_t ld, int64_t col0,
                                           int tid) {
  constexpr int P = XPitch<T>::value;
  constexpr int V = 16 / sizeof(T);             // elements per 16-byte copy
  constexpr int PER_ROW = kRC / V;              // copies per row
  for (int i = tid; i < kRT * PER_ROW; i += kRThreads) {
    const int r = i / PER_ROW, c = (i % PER_ROW) * V;
    const bool ok = row0 + r < nrows;
    cp16(saddr(dst + r * P + c), ok ? (const void*)(src + (row0 + r) * ld + col0 + c) : (const void*)src, ok);
  }
}

// rows k0..k0+63 of Wr (d,E) as 64 x EP fp32, experts >= E zero (16-byte
// copies when every row of Wr starts on a 16-byte boundary, else 4-byte)
template <int EP>
__device__ __forceinline__ void stage_wr(float* dst, const float* Wr, int k0, int E, int tid) {
  if ((E & 3) == 0 && (reinterpret_cast<uintptr_t>(Wr) & 15u) == 0) {
    constexpr int PER_ROW = EP / 4;
    for (int i = tid; i < kRC * PER_ROW; i += kRThreads) {
      const int r = i / PER_ROW, c = (i % PER_ROW) * 4;
      const bool ok = c < E;
      cp16(saddr(dst + r * EP + c), ok ? (const void*)(Wr + (int64_t)(k0 + r) * E + c) : (const void*)Wr, ok);
    }
  } else {
    for (int i = tid; i < kRC * EP; i += kRThreads) {
      const int r = i / EP, c = i % EP;
      const bool ok = c < E;
      cp4(saddr(dst + r * EP + c), ok ? (const void*)(Wr + (int64_t)(k0 + r) * E + c) : (const void*)Wr, ok);
    }
  }
}

// ------------------------------------------------------------------ forward
template <typename T, int EP>
__global__ void __launch_bounds__(kRThreads) router_fwd_kernel(const T* __restrict__ x, const float* __restrict__ Wr,
                                                               const float* __restrict__ bias, int64_t L, int d, int E,
                                                               int K, int32_t* __restrict__ ids,
                                                               float* __restrict__ gates) {
  using Ly = RLayout<EP>;
  constexpr int S = Ly::STAGES, P = XPitch<T>::value;
  constexpr int XS = kRT * P;  // elements of one x stage
  extern __shared__ __align__(16) uint8_t rsm[];
  T* xs = reinterpret_cast<T*>(rsm);
  float* ws = reinterpret_cast<float*>(rsm + S * XS * sizeof(T));
  const int tid = threadIdx.x, te = tid % Ly::TE, tr = tid / Ly::TE;
  const int64_t t0 = (int64_t)blockIdx.x * kRT;
  const int nch = d / kRC;
  float acc[Ly::RPT][Ly::EPT];
#pragma unroll
  for (int i = 0; i < Ly::RPT; ++i)
#pragma unroll
    for (int j = 0; j < Ly::EPT; ++j) acc[i][j] = 0.f;

#pragma unroll
  for (int c = 0; c < S - 1; ++c) {
    if (c < nch) {
      stage_rows<T>(xs + c * XS, x, t0, L, d, (int64_t)c * kRC, tid);
      stage_wr<EP>(ws + c * kRC * EP, Wr, c * kRC, E, tid);
    }
    cp_commit();
  }
  for (int c = 0; c < nch; ++c) {
    cp_wait<S - 2>();
    __syncthreads();
    {  // the chunk S-1 ahead goes into the stage that chunk c-1 used
      const int n = c + S - 1;
      if (n < nch) {
        stage_rows<T>(xs + (n % S) * XS, x, t0, L, d, (int64_t)n * kRC, tid);
        stage_wr<EP>(ws + (n % S) * kRC * EP, Wr, n * kRC, E, tid);
      }
      cp_commit();
    }
    const T* xa = xs + (c % S) * XS;
    const float* wb = ws + (c % S) * kRC * EP;
#pragma unroll 4
    for (int k = 0; k < kRC; ++k) {
      float av[Ly::RPT], bv[Ly::EPT];
#pragma unroll
      for (int i = 0; i < Ly::RPT; ++i) av[i] = to_f32(xa[(tr * Ly::RPT + i) * P + k]);
#pragma unroll
      for (int j = 0; j < Ly::EPT; ++j) bv[j] = wb[k * EP + j * Ly::TE + te];
#pragma unroll
      for (int i = 0; i < Ly::RPT; ++i)
#pragma unroll
        for (int j = 0; j < Ly::EPT; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
  cp_wait<0>();

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

// Forward for few experts (EP <= 16) when Wr fits in shared memory: a
// GEMV over the token rows.  Wr (d, EP) is staged once per CTA; each warp
// takes 4 tokens at a time, its lanes read 16-byte pieces of the 4 rows
// (columns lane*8 + 256*i) and accumulate 4 x EP partial logits, which a
// butterfly reduction completes; lane k of the warp then ranks token k's
// logits (larger first, equal to the lower index) and writes its ids and
// gates.  The x rows stream from HBM once, coalesced.
template <typename T, int EP>
__global__ void __launch_bounds__(512) router_fwd_gemv_kernel(const T* __restrict__ x, const float* __restrict__ Wr,
                                                              const float* __restrict__ bias, int64_t L, int d, int E,
                                                              int K, int32_t* __restrict__ ids,
                                                              float* __restrict__ gates) {
  constexpr int TPW = 4;  // tokens per warp pass
  extern __shared__ __align__(16) uint8_t rsm[];
  // Wr as [d][EP] with 4 floats of padding after every 8 rows: the lanes of
  // a warp read rows 8 apart, which then fall on different banks
  float* ws = reinterpret_cast<float*>(rsm);
  for (int i = threadIdx.x; i < d * EP; i += blockDim.x) {
    const int r = i / EP, c = i % EP;
    const bool ok = c < E;
    cp4(saddr(ws + r * EP + (r >> 3) * 4 + c), ok ? (const void*)(Wr + (int64_t)r * E + c) : (const void*)Wr, ok);
  }
  cp_commit();
  cp_wait<0>();
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t0 = warp * TPW; t0 < L; t0 += nwarps * TPW) {
    // pairs of experts per packed fp32x2 FMA for up to 8 experts (each half
    // is an ordinary fp32 FMA, round to nearest, so the logits are the same)
    float2 acc2[TPW][EP / 2];
#pragma unroll
    for (int q = 0; q < TPW; ++q)
#pragma unroll
      for (int e = 0; e < EP / 2; ++e) acc2[q][e] = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
      float xv[TPW][8];
#pragma unroll
      for (int q = 0; q < TPW; ++q) {
        if (t0 + q < L) {
          load8(x + (t0 + q) * d + c0, xv[q]);
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) xv[q][u] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4* wr = reinterpret_cast<const float4*>(ws + (c0 + u) * EP + (c0 >> 3) * 4);
#pragma unroll
        for (int e4 = 0; e4 < EP / 4; ++e4) {
          const float4 w = wr[e4];
          const float2 wa = make_float2(w.x, w.y), wb = make_float2(w.z, w.w);
#pragma unroll
          for (int q = 0; q < TPW; ++q) {
            const float2 x2 = make_float2(xv[q][u], xv[q][u]);
            if constexpr (EP <= 8) {
              acc2[q][2 * e4 + 0] = __ffma2_rn(x2, wa, acc2[q][2 * e4 + 0]);
              acc2[q][2 * e4 + 1] = __ffma2_rn(x2, wb, acc2[q][2 * e4 + 1]);
            } else {  // 16 experts: scalar FMAs keep the registers within the 512-thread budget
              acc2[q][2 * e4 + 0].x = fmaf(x2.x, wa.x, acc2[q][2 * e4 + 0].x);
              acc2[q][2 * e4 + 0].y = fmaf(x2.x, wa.y, acc2[q][2 * e4 + 0].y);
              acc2[q][2 * e4 + 1].x = fmaf(x2.x, wb.x, acc2[q][2 * e4 + 1].x);
              acc2[q][2 * e4 + 1].y = fmaf(x2.x, wb.y, acc2[q][2 * e4 + 1].y);
            }
          }
        }
      }
    }
    float acc[TPW][EP];
#pragma unroll
    for (int q = 0; q < TPW; ++q)
#pragma unroll
      for (int e = 0; e < EP / 2; ++e) {
        acc[q][2 * e] = acc2[q][e].x;
        acc[q][2 * e + 1] = acc2[q][e].y;
      }
#pragma unroll
    for (int q = 0; q < TPW; ++q)
#pragma unroll
      for (int e = 0; e < EP; ++e)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[q][e] += __shfl_xor_sync(0xffffffffu, acc[q][e], off);
    // lane q ranks token t0 + q
#pragma unroll
    for (int q = 0; q < TPW; ++q) {
      const int64_t t = t0 + q;
      if (lane != q || t >= L) continue;
      float lg[EP];
#pragma unroll
      for (int e = 0; e < EP; ++e) lg[e] = e < E ? acc[q][e] + (bias ? bias[e] : 0.f) : -FLT_MAX;
      uint32_t taken = 0;
      float selv[kMaxK], w[kMaxK], sum = 0.f;
      int seli[kMaxK];
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        selv[k] = 0.f;
        seli[k] = 0;
        if (k < K) {
          float bv = -FLT_MAX;
          int bi = INT_MAX;
#pragma unroll
          for (int e = 0; e < EP; ++e)
            if (!((taken >> e) & 1u) && e < E && (lg[e] > bv || (lg[e] == bv && e < bi))) {
              bv = lg[e];
              bi = e;
            }
          selv[k] = bv;
          seli[k] = bi;
          taken |= 1u << bi;
        }
      }
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
// dx = dlogit Wr^T for one 64-token tile, Wr streamed in 64-row chunks
template <typename T, int EP>
__global__ void __launch_bounds__(kRThreads) router_dx_kernel(const float* __restrict__ Wr,
                                                              const int32_t* __restrict__ ids,
                                                              const float* __restrict__ gates,
                                                              const float* __restrict__ dgates, int64_t L, int d, int E,
                                                              int K, float* __restrict__ dl, T* __restrict__ dx) {
  constexpr int S = 3;
  __shared__ float dls[kRT][kMaxK];
  __shared__ int ids_s[kRT][kMaxK];
  extern __shared__ __align__(16) uint8_t rsm[];
  float* ws = reinterpret_cast<float*>(rsm);  // S stages of 64 x EP
  const int tid = threadIdx.x;
  const int64_t t0 = (int64_t)blockIdx.x * kRT;
  const int nch = d / kRC;
  if (dx) {
#pragma unroll
    for (int c = 0; c < S - 1; ++c) {
      if (c < nch) stage_wr<EP>(ws + c * kRC * EP, Wr, c * kRC, E, tid);
      cp_commit();
    }
  }
  if (tid < kRT) {
    const int64_t t = t0 + tid;
    float g[kMaxK], dg[kMaxK], s = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      g[k] = (k < K && t < L) ? gates[t * K + k] : 0.f;
      dg[k] = (k < K && t < L) ? dgates[t * K + k] : 0.f;
      const int e = (k < K && t < L) ? ids[t * K + k] : 0;
      ids_s[tid][k] = ((unsigned)e < (unsigned)E) ? e : 0;
      s = fmaf(g[k], dg[k], s);
    }
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      const float v = g[k] * (dg[k] - s);
      dls[tid][k] = k < K ? v : 0.f;
      if (k < K && t < L) dl[t * K + k] = v;
    }
  }
  if (!dx) return;
  const int row = tid >> 2, c16 = (tid & 3) * 16;  // 16 outputs of one token per thread
  for (int c = 0; c < nch; ++c) {
    cp_wait<S - 2>();
    __syncthreads();
    {
      const int n = c + S - 1;
      if (n < nch) stage_wr<EP>(ws + (n % S) * kRC * EP, Wr, n * kRC, E, tid);
      cp_commit();
    }
    const float* wb = ws + (c % S) * kRC * EP;
    float out[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) out[u] = 0.f;
    for (int k = 0; k < K; ++k) {  // the slot's dlogit and expert column, hoisted
      const float dv = dls[row][k];
      const float* wcol = wb + c16 * EP + ids_s[row][k];
#pragma unroll
      for (int u = 0; u < 16; ++u) out[u] = fmaf(dv, wcol[u * EP], out[u]);
    }
    if (t0 + row < L) {
      T* o = dx + (t0 + row) * d + (int64_t)c * kRC + c16;
      store8(o, out);
      store8(o + 8, out + 8);
    }
  }
  cp_wait<0>();
}

// partial dWr (and dbias) of one 64-row block of Wr over one token split:
// part[s][j][e] = sum_{t in split s} x[t, j] dlogit[t, e].  Each 64-token
// chunk stages x[t, j0..j0+63] and the chunk's ids and dlogits by cp.async,
// then expands the dlogits into a dense 64 x EP tile.
template <typename T, int EP>
__global__ void __launch_bounds__(kRThreads) router_dwr_kernel(const T* __restrict__ x, const int32_t* __restrict__ ids,
                                                               const float* __restrict__ dl, int64_t L, int d, int E,
                                                               int K, int64_t split, float* __restrict__ part,
                                                               float* __restrict__ part_b) {
  using Ly = RLayout<EP>;
  constexpr int S = 3, P = XPitch<T>::value;
  constexpr int XS = kRT * P;
  extern __shared__ __align__(16) uint8_t rsm[];
  T* xs = reinterpret_cast<T*>(rsm);                                            // S x [64 tokens][P]
  float* dd = reinterpret_cast<float*>(rsm + S * XS * sizeof(T));              // [64 tokens][EP]
  int32_t* is = reinterpret_cast<int32_t*>(dd + kRT * EP);                     // S x [64 * kMaxK]
  float* ls = reinterpret_cast<float*>(is + S * kRT * kMaxK);                  // S x [64 * kMaxK]
  const int tid = threadIdx.x, te = tid % Ly::TE, tr = tid / Ly::TE;
  const int j0 = blockIdx.x * kRT;
  const int64_t ts = (int64_t)blockIdx.y * split;
  const int64_t tend = min(L, ts + split);
  const int nch = (int)((tend - ts + kRT - 1) / kRT);
  float acc[Ly::RPT][Ly::EPT];
#pragma unroll
  for (int i = 0; i < Ly::RPT; ++i)
#pragma unroll
    for (int j = 0; j < Ly::EPT; ++j) acc[i][j] = 0.f;
  float bacc = 0.f;
  auto stage = [&](int c) {
    const int st = c % S;
    const int64_t c0 = ts + (int64_t)c * kRT;
    stage_rows<T>(xs + st * XS, x, c0, tend, d, j0, tid);
    for (int i = tid; i < kRT * K; i += kRThreads) {
      const bool ok = c0 * K + i < tend * K;
      cp4(saddr(is + st * kRT * kMaxK + i), ok ? (const void*)(ids + c0 * K + i) : (const void*)ids, ok);
      cp4(saddr(ls + st * kRT * kMaxK + i), ok ? (const void*)(dl + c0 * K + i) : (const void*)dl, ok);
    }
  };
#pragma unroll
  for (int c = 0; c < S - 1; ++c) {
    if (c < nch) stage(c);
    cp_commit();
  }
  for (int c = 0; c < nch; ++c) {
    cp_wait<S - 2>();
    __syncthreads();  // chunk c landed; every thread is done with chunk c-1 and its dense tile
    {
      const int n = c + S - 1;
      if (n < nch) stage(n);
      cp_commit();
    }
    const int st = c % S;
    for (int i = tid; i < kRT * EP; i += kRThreads) dd[i] = 0.f;
    __syncthreads();
    if (tid < kRT) {
      for (int k = 0; k < K; ++k) {
        const int e = is[st * kRT * kMaxK + tid * K + k];
        if ((unsigned)e < (unsigned)E) dd[tid * EP + e] = ls[st * kRT * kMaxK + tid * K + k];
      }
    }
    __syncthreads();
    const T* xa = xs + st * XS;
#pragma unroll 4
    for (int t = 0; t < kRT; ++t) {
      float av[Ly::RPT], bv[Ly::EPT];
#pragma unroll
      for (int i = 0; i < Ly::RPT; ++i) av[i] = to_f32(xa[t * P + tr * Ly::RPT + i]);
#pragma unroll
      for (int j = 0; j < Ly::EPT; ++j) bv[j] = dd[t * EP + j * Ly::TE + te];
#pragma unroll
      for (int i = 0; i < Ly::RPT; ++i)
#pragma unroll
        for (int j = 0; j < Ly::EPT; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (blockIdx.x == 0 && tid < EP) {
      for (int t = 0; t < kRT; ++t) bacc += dd[t * EP + tid];
    }
  }
  cp_wait<0>();
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

// The router backward for few experts (EP <= 16) in one pass over x: a
// thread owns 8 consecutive columns j of x (rows of Wr) for all EP experts.
// Per 64-token chunk the first 64 threads form the chunk's dlogits (the
// softmax over the selected logits: dl_k = g_k (dg_k - sum_i g_i dg_i)),
// as a dense 64 x EP tile and per slot; every thread then, token by token,
// writes dx[t, j..j+7] = sum_k dl_k Wr[j.., e_k] (the CTA's rows of Wr
// staged transposed in shared memory, so a thread's 8 values of one expert
// are 32 contiguous bytes) and adds x[t, j..j+7] dl[t, :] to its partial
// dWr.  Each thread keeps its next kBwAhead pieces of x in flight by
// cp.async into a ring of its own in shared memory.  part[s][j][e] = sum over the split's tokens, summed in a fixed order
// by router_reduce_kernel.
constexpr int kBwThreads = 128;
constexpr int kBwCols = kBwThreads * 8;  // columns of x (rows of Wr) per CTA
constexpr int kBwAhead = 8;              // tokens of x each thread has in flight (cp.async)
template <typename T, int EP>
constexpr size_t bwd_small_smem() {
  return (size_t)EP * kBwCols * sizeof(float) + (size_t)kBwAhead * kBwThreads * 8 * sizeof(T);
}

template <typename T, int EP>
__global__ void __launch_bounds__(kBwThreads) router_bwd_small_kernel(
    const T* __restrict__ x, const float* __restrict__ Wr, const int32_t* __restrict__ ids,
    const float* __restrict__ gates, const float* __restrict__ dgates, int64_t L, int d, int E, int K, int64_t split,
    T* __restrict__ dx, float* __restrict__ part, float* __restrict__ part_b) {
  extern __shared__ __align__(16) uint8_t rsm[];
  float* wt = reinterpret_cast<float*>(rsm);  // [EP][kBwCols]: Wr^T, this CTA's columns
  T* xs = reinterpret_cast<T*>(wt + EP * kBwCols);  // [kBwAhead][kBwThreads][8]: each thread's own x pieces
  __shared__ __align__(16) float dd[kRT][EP];
  __shared__ float dls[kRT][kMaxK];
  __shared__ int ids_s[kRT][kMaxK];
  const int tid = threadIdx.x;
  const int col0 = blockIdx.x * kBwCols;
  const int j = col0 + tid * 8;
  const bool jv = j < d;
  for (int i = tid; i < EP * kBwCols; i += kBwThreads) {
    const int e = i / kBwCols, c = i % kBwCols;
    wt[i] = (e < E && col0 + c < d) ? Wr[(int64_t)(col0 + c) * E + e] : 0.f;
  }
  const int64_t ts = (int64_t)blockIdx.y * split;
  const int64_t tend = min(L, ts + split);
  float acc[8][EP];
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[u][e] = 0.f;
  float bacc = 0.f;
  for (int64_t c0 = ts; c0 < tend; c0 += kRT) {
    __syncthreads();  // every thread is done with the previous chunk's dlogits
    if (tid < kRT) {
      const int64_t t = c0 + tid;
      const bool tv = t < tend;
      float g[kMaxK], dg[kMaxK], sdot = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        g[k] = (k < K && tv) ? gates[t * K + k] : 0.f;
        dg[k] = (k < K && tv) ? dgates[t * K + k] : 0.f;
        const int e = (k < K && tv) ? ids[t * K + k] : 0;
        ids_s[tid][k] = ((unsigned)e < (unsigned)E) ? e : 0;
        sdot = fmaf(g[k], dg[k], sdot);
      }
#pragma unroll
      for (int e = 0; e < EP; ++e) dd[tid][e] = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        const float v = g[k] * (dg[k] - sdot);
        dls[tid][k] = k < K ? v : 0.f;
        if (k < K && tv) {
          const int e = ids[t * K + k];
          if ((unsigned)e < (unsigned)E) dd[tid][e] = v;
        }
      }
    }
    __syncthreads();
    const int n = (int)min((int64_t)kRT, tend - c0);
    if (blockIdx.x == 0 && tid < EP)
      for (int t = 0; t < n; ++t) bacc += dd[t][tid];
    if (!jv) continue;
    // the thread's 8 columns of token c0 + tt into its own ring slot tt % kBwAhead
    auto fetch = [&](int tt) {
      const T* src = x + (c0 + tt) * d + j;
      const uint32_t dst = saddr(xs + ((tt % kBwAhead) * kBwThreads + tid) * 8);
#pragma unroll
      for (int q = 0; q < (int)(8 * sizeof(T) / 16); ++q) cp16(dst + 16 * q, src + q * (16 / sizeof(T)), true);
    };
#pragma unroll
    for (int tt = 0; tt < kBwAhead; ++tt) {
      if (tt < n) fetch(tt);
      cp_commit();
    }
    for (int t = 0; t < n; ++t) {
      cp_wait<kBwAhead - 1>();  // token t's copy (groups complete in order) has landed
      float xv[8];
      load8(xs + ((t % kBwAhead) * kBwThreads + tid) * 8, xv);
      if (t + kBwAhead < n) fetch(t + kBwAhead);
      cp_commit();
      if (dx) {
        float out[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) out[u] = 0.f;
        for (int k = 0; k < K; ++k) {
          const float dv = dls[t][k];
          const float4* wr = reinterpret_cast<const float4*>(wt + ids_s[t][k] * kBwCols + tid * 8);
          const float4 w0 = wr[0], w1 = wr[1];
          out[0] = fmaf(dv, w0.x, out[0]);
          out[1] = fmaf(dv, w0.y, out[1]);
          out[2] = fmaf(dv, w0.z, out[2]);
          out[3] = fmaf(dv, w0.w, out[3]);
          out[4] = fmaf(dv, w1.x, out[4]);
          out[5] = fmaf(dv, w1.y, out[5]);
          out[6] = fmaf(dv, w1.z, out[6]);
          out[7] = fmaf(dv, w1.w, out[7]);
        }
        store8(dx + (c0 + t) * d + j, out);
      }
      const float4* dr = reinterpret_cast<const float4*>(&dd[t][0]);
#pragma unroll
      for (int e4 = 0; e4 < EP / 4; ++e4) {
        const float4 w = dr[e4];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc[u][4 * e4 + 0] = fmaf(xv[u], w.x, acc[u][4 * e4 + 0]);
          acc[u][4 * e4 + 1] = fmaf(xv[u], w.y, acc[u][4 * e4 + 1]);
          acc[u][4 * e4 + 2] = fmaf(xv[u], w.z, acc[u][4 * e4 + 2]);
          acc[u][4 * e4 + 3] = fmaf(xv[u], w.w, acc[u][4 * e4 + 3]);
        }
      }
    }
  }
  float* dst = part + (int64_t)blockIdx.y * d * E;
  if (jv) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (e < E) dst[(int64_t)(j + u) * E + e] = acc[u][e];
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

// column blocks of the dWr kernel: 64 rows of Wr per CTA, or for few
// experts 8 rows per thread of a 256-thread CTA
int64_t router_col_blocks(const moeblaze_shape& s) {
  return padded_experts(s.E) <= 16 ? (s.d + kBwCols - 1) / kBwCols : s.d / kRT;
}

// token splits of the weight-gradient sums: enough CTAs to fill the GPU a
// few times over, at least one 64-token chunk per split
int64_t router_splits(const moeblaze_shape& s) {
  const int64_t jb = router_col_blocks(s);
  int64_t S = (4 * (int64_t)sm_count() + jb - 1) / jb;
  const int64_t chunks = (s.L + kRT - 1) / kRT;
  if (S > chunks) S = chunks;
  return S < 1 ? 1 : S;
}

template <typename T, int EP>
size_t fwd_smem() {
  return RLayout<EP>::STAGES * ((size_t)kRT * XPitch<T>::value * sizeof(T) + (size_t)kRC * EP * sizeof(float));
}
template <int EP>
size_t dx_smem() {
  return 3 * (size_t)kRC * EP * sizeof(float);
}
template <typename T, int EP>
size_t dwr_smem() {
  return 3 * (size_t)kRT * XPitch<T>::value * sizeof(T) + (size_t)kRT * EP * sizeof(float) +
         3 * 2 * (size_t)kRT * kMaxK * 4;
}

constexpr size_t kGemvWrBytes = 160 * 1024;  // largest Wr staged whole by the GEMV forward

template <typename T, int EP>
moeblaze_status fwd_ep(const moeblaze_shape& s, const void* x, const float* Wr, const float* bias, int32_t* ids,
                       float* gates, cudaStream_t st) {
  if constexpr (EP <= 16) {
    const size_t wb = ((size_t)s.d * EP + (size_t)s.d / 2) * sizeof(float);
    if (wb <= kGemvWrBytes) {
      auto kern = router_fwd_gemv_kernel<T, EP>;
      MB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wb));
      const int threads = 512;
      int64_t blocks = (s.L + (threads / 32) * 4 - 1) / ((threads / 32) * 4);
      if (blocks > (int64_t)sm_count()) blocks = sm_count();  // one persistent CTA per SM
      kern<<<(unsigned)blocks, threads, wb, st>>>(static_cast<const T*>(x), Wr, bias, s.L, s.d, s.E, s.K, ids, gates);
      MB_CUDA(cudaGetLastError());
      count_launch();
      return MOEBLAZE_OK;
    }
  }
  auto kern = router_fwd_kernel<T, EP>;
  const size_t sm = fwd_smem<T, EP>();
  MB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
  const unsigned grid = (unsigned)((s.L + kRT - 1) / kRT);
  kern<<<grid, kRThreads, sm, st>>>(static_cast<const T*>(x), Wr, bias, s.L, s.d, s.E, s.K, ids, gates);
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

template <typename T, int EP>
moeblaze_status bwd_ep(const moeblaze_shape& s, const void* x, const float* Wr, const int32_t* ids,
                       const float* gates, const float* dgates, float* dWr, float* dbias, void* dx, void* ws,
                       cudaStream_t st) {
  const int64_t S = router_splits(s);
  const int64_t split = ((s.L + S - 1) / S + kRT - 1) / kRT * kRT;
  char* w = static_cast<char*>(ws);
  float* dl = reinterpret_cast<float*>(w);
  float* part = reinterpret_cast<float*>(w + align_up(sizeof(float) * s.L * s.K, 256));
  float* part_b = part + (size_t)S * s.d * s.E;
  if constexpr (EP <= 16) {
    auto kern = router_bwd_small_kernel<T, EP>;
    const size_t sm = bwd_small_smem<T, EP>();  // plus 6 KB of static shared memory: always above the default limit
    MB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
    kern<<<dim3((unsigned)router_col_blocks(s), (unsigned)S), kBwThreads, sm, st>>>(
        static_cast<const T*>(x), Wr, ids, gates, dgates, s.L, s.d, s.E, s.K, split, static_cast<T*>(dx), part,
        part_b);
    MB_CUDA(cudaGetLastError());
    count_launch();
  } else {
    const unsigned tiles = (unsigned)((s.L + kRT - 1) / kRT);
    {
      auto kern = router_dx_kernel<T, EP>;
      const size_t sm = dx_smem<EP>();
      MB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
      kern<<<tiles, kRThreads, sm, st>>>(Wr, ids, gates, dgates, s.L, s.d, s.E, s.K, dl, static_cast<T*>(dx));
      MB_CUDA(cudaGetLastError());
    }
    auto kern = router_dwr_kernel<T, EP>;
    const size_t sm = dwr_smem<T, EP>();
    MB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
    kern<<<dim3((unsigned)(s.d / kRT), (unsigned)S), kRThreads, sm, st>>>(static_cast<const T*>(x), ids, dl, s.L, s.d,
                                                                          s.E, s.K, split, part, part_b);
    MB_CUDA(cudaGetLastError());
    count_launch(2);
  }
  const int64_t n = (int64_t)s.d * s.E;
  int64_t blocks = (n + s.E + 255) / 256;
  if (blocks > 8 * (int64_t)sm_count()) blocks = 8 * (int64_t)sm_count();
  router_reduce_kernel<<<(unsigned)blocks, 256, 0, st>>>(part, part_b, n, s.E, (int)S, dWr, dbias);
  MB_CUDA(cudaGetLastError());
  count_launch();
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
