// fp32 path of the layer: the same stages, index structures and fused
// epilogues as the bf16 tensor-core path, with fp32 storage and fp32 FFMA
// arithmetic on CUDA cores (TF32 tensor cores would not hold the fp32
// tolerance).  Meant for small fp32 layers; one 16x16 output tile per CTA,
// operands staged through shared memory.
//
// Row space: every expert's routed rows occupy a segment of the padded row
// space [pad_off[e], pad_off[e+1]), a multiple of 256 rows; row q of expert e
// with i = q - pad_off[e] < n_e is routed row p = off[e] + i of token
// D1[p].  Padding rows compute on a valid token (so every gathered address is
// in bounds) and are written as zeros where they feed a reduction.
#include "common.cuh"

namespace moeblaze {
namespace {

constexpr int T = 16;

struct RowCtx {
  int e;        // expert of the tile, -1 if the tile is past the end
  int q0;       // first padded row of the tile
  int pad0;     // pad_off[e]
  int n;        // n_e
  int off;      // expert_token_offsets[e]
};

struct Common {
  const int32_t* D1;
  const int32_t* D2;
  const int32_t* D3;
  const float* gates;
  MetaView meta;
  int64_t L;
  int d, h, E, K;

  __device__ bool row_ctx(int mt16, RowCtx& c) const {
    c.q0 = mt16 * T;
    const int m128 = c.q0 / kTileM;
    if (m128 >= *meta.num_m_tiles) return false;
    c.e = meta.tile_expert[m128];
    if (c.e < 0) return false;
    c.pad0 = meta.pad_off[c.e];
    c.off = D2[c.e];
    c.n = D2[c.e + 1] - c.off;
    return true;
  }
  // token of padded row q (clamped to the expert's last routed row)
  __device__ int token(const RowCtx& c, int q) const {
    int i = q - c.pad0;
    if (i >= c.n) i = c.n - 1;
    return D1[c.off + i];
  }
  __device__ bool valid(const RowCtx& c, int q) const { return q - c.pad0 < c.n; }
  // the dispatch was built for this call's (L, E, K); otherwise record the
  // mismatch and read nothing of it (the same answer in every thread)
  __device__ bool shape_ok() const {
    if (meta_matches(meta.hdr, L, E, K)) return true;
    if (threadIdx.x == 0 && threadIdx.y == 0) atomicOr(meta.err, kErrShapeMismatch);
    return false;
  }
  __device__ float gate(int t, int e, int* slot = nullptr) const {
    for (int k = 0; k < K; ++k)
      if (D3[(int64_t)t * K + k] == e) {
        if (slot) *slot = k;
        return gates[(int64_t)t * K + k];
      }
    if (slot) *slot = 0;
    return 0.f;
  }
};

// ------------------------------------------------------------- up projection
// A = x[tok] W1_e, B = x[tok] W2_e (SwiGLU) ; H = SiLU(A) * B  (SiLU: H = SiLU(A))
__global__ void up_kernel(Common c, const float* __restrict__ x, const float* __restrict__ W1,
                          const float* __restrict__ W2, float* __restrict__ A, float* __restrict__ B,
                          float* __restrict__ H, int64_t rows, bool swiglu) {
  if (!c.shape_ok()) return;
  __shared__ float Xs[T][T + 1], W1s[T][T + 1], W2s[T][T + 1];
  __shared__ int toks[T];
  RowCtx r;
  if (!c.row_ctx(blockIdx.x, r)) return;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int q = r.q0 + ty, j = blockIdx.y * T + tx;
  if (ty == 0) toks[tx] = c.token(r, r.q0 + tx);
  __syncthreads();
  float a = 0.f, b = 0.f;
  for (int k0 = 0; k0 < c.d; k0 += T) {
    const int ka = k0 + tx, kb = k0 + ty;
    Xs[ty][tx] = ka < c.d ? x[(int64_t)toks[ty] * c.d + ka] : 0.f;
    const bool okb = kb < c.d && j < c.h;
    W1s[ty][tx] = okb ? W1[((int64_t)r.e * c.d + kb) * c.h + j] : 0.f;
    if (swiglu) W2s[ty][tx] = okb ? W2[((int64_t)r.e * c.d + kb) * c.h + j] : 0.f;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < T; ++kk) {
      a = fmaf(Xs[ty][kk], W1s[kk][tx], a);
      if (swiglu) b = fmaf(Xs[ty][kk], W2s[kk][tx], b);
    }
    __syncthreads();
  }
  if (j >= c.h) return;
  const bool ok = c.valid(r, q);
  const int64_t o = (int64_t)q * c.h + j;
  const float s = a / (1.f + expf(-a));
  A[o] = ok ? a : 0.f;
  if (swiglu) B[o] = ok ? b : 0.f;
  H[o] = ok ? (swiglu ? s * b : s) : 0.f;
  (void)rows;
}

// ------------------------------------------------------- down + fused combine
// y[t] += g * (H W3_e)[row]
__global__ void down_kernel(Common c, const float* __restrict__ H, const float* __restrict__ W3,
                            float* __restrict__ y) {
  if (!c.shape_ok()) return;
  __shared__ float Hs[T][T + 1], Ws[T][T + 1];
  RowCtx r;
  if (!c.row_ctx(blockIdx.x, r)) return;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int q = r.q0 + ty, col = blockIdx.y * T + tx;
  float acc = 0.f;
  for (int k0 = 0; k0 < c.h; k0 += T) {
    const int ka = k0 + tx, kb = k0 + ty;
    Hs[ty][tx] = ka < c.h ? H[(int64_t)q * c.h + ka] : 0.f;
    Ws[ty][tx] = (kb < c.h && col < c.d) ? W3[((int64_t)r.e * c.h + kb) * c.d + col] : 0.f;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < T; ++kk) acc = fmaf(Hs[ty][kk], Ws[kk][tx], acc);
    __syncthreads();
  }
  if (col >= c.d || !c.valid(r, q)) return;
  const int t = c.token(r, q);
  atomicAdd(&y[(int64_t)t * c.d + col], c.gate(t, r.e) * acc);
}

// ------------------------------------------- dH = g dY[t] W3_e^T + SwiGLU bwd
// dA = dH * B * SiLU'(A), dB = dH * SiLU(A), Hg = g * SiLU(A) * B
__global__ void dh_kernel(Common c, const float* __restrict__ dY, const float* __restrict__ W3,
                          const float* __restrict__ A, const float* __restrict__ B, float* __restrict__ dAB,
                          float* __restrict__ Hg, float* __restrict__ dg, bool swiglu) {
  if (!c.shape_ok()) return;
  __shared__ float Gs[T][T + 1], Ws[T][T + 1];
  __shared__ int toks[T];
  RowCtx r;
  if (!c.row_ctx(blockIdx.x, r)) return;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int q = r.q0 + ty, j = blockIdx.y * T + tx;
  if (ty == 0) toks[tx] = c.token(r, r.q0 + tx);
  __syncthreads();
  float acc = 0.f;
  for (int k0 = 0; k0 < c.d; k0 += T) {
    const int ka = k0 + tx;
    Gs[ty][tx] = ka < c.d ? dY[(int64_t)toks[ty] * c.d + ka] : 0.f;
    // Ws[kk][n] = W3[e][n][k]: element (k = k0+ty, n = j-col tx) loaded transposed
    const int jn = blockIdx.y * T + ty, kc = k0 + tx;
    Ws[tx][ty] = (jn < c.h && kc < c.d) ? W3[((int64_t)r.e * c.h + jn) * c.d + kc] : 0.f;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < T; ++kk) acc = fmaf(Gs[ty][kk], Ws[kk][tx], acc);
    __syncthreads();
  }
  if (j >= c.h) return;
  const int nb = swiglu ? 2 : 1;
  const int64_t o = (int64_t)q * c.h + j;
  const int64_t oab = (int64_t)q * nb * c.h + j;
  if (!c.valid(r, q)) {
    dAB[oab] = 0.f;
    if (swiglu) dAB[oab + c.h] = 0.f;
    Hg[o] = 0.f;
    return;
  }
  const int t = toks[ty];
  int kslot = 0;
  const float g = c.gate(t, r.e, &kslot);
  const float dH = g * acc;
  const float a = A[o];
  const float sg = 1.f / (1.f + expf(-a));
  const float s = a * sg;
  const float dsilu = sg * (1.f + a * (1.f - sg));
  if (swiglu) {
    const float b = B[o];
    dAB[oab] = dH * b * dsilu;
    dAB[oab + c.h] = dH * s;
    Hg[o] = g * s * b;
    if (dg) atomicAdd(&dg[(int64_t)t * c.K + kslot], s * b * acc);  // <H_row, dY W3^T>
  } else {
    dAB[oab] = dH * dsilu;
    Hg[o] = g * s;
    if (dg) atomicAdd(&dg[(int64_t)t * c.K + kslot], s * acc);
  }
}

// ------------------------------------------------ dX = dA W1^T + dB W2^T, combine
__global__ void dx_kernel(Common c, const float* __restrict__ dAB, const float* __restrict__ W1,
                          const float* __restrict__ W2, float* __restrict__ dX, bool swiglu) {
  if (!c.shape_ok()) return;
  __shared__ float As[T][T + 1], Ws[T][T + 1];
  RowCtx r;
  if (!c.row_ctx(blockIdx.x, r)) return;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int q = r.q0 + ty, col = blockIdx.y * T + tx;
  const int nb = swiglu ? 2 : 1;
  const int Kd = nb * c.h;
  float acc = 0.f;
  for (int k0 = 0; k0 < Kd; k0 += T) {
    const int ka = k0 + tx;
    As[ty][tx] = ka < Kd ? dAB[(int64_t)q * Kd + ka] : 0.f;
    // Ws[kk][n] = W{1,2}[e][n][k mod h]
    const int cn = blockIdx.y * T + ty, kc = k0 + tx;
    float w = 0.f;
    if (cn < c.d && kc < Kd) {
      const float* W = kc < c.h ? W1 : W2;
      const int kk = kc < c.h ? kc : kc - c.h;
      w = W[((int64_t)r.e * c.d + cn) * c.h + kk];
    }
    Ws[tx][ty] = w;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < T; ++kk) acc = fmaf(As[ty][kk], Ws[kk][tx], acc);
    __syncthreads();
  }
  if (col >= c.d || !c.valid(r, q)) return;
  const int t = c.token(r, q);
  atomicAdd(&dX[(int64_t)t * c.d + col], acc);
}

// --------------------------------------------------------- weight gradients
// dW1_e[i][j] = sum_q x[tok q][i] dA[q][j] ; dW2 with dB ; over the expert's rows
__global__ void dw12_kernel(Common c, const float* __restrict__ x, const float* __restrict__ dAB,
                            float* __restrict__ dW1, float* __restrict__ dW2, bool swiglu) {
  if (!c.shape_ok()) return;
  __shared__ float Xs[T][T + 1], As[T][T + 1], Bs[T][T + 1];
  __shared__ int toks[T];
  const int e = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int i = blockIdx.x * T + ty, j = blockIdx.y * T + tx;
  const int pad0 = c.meta.pad_off[e], pad1 = c.meta.pad_off[e + 1];
  const int off = c.D2[e], n = c.D2[e + 1] - off;
  const int nb = swiglu ? 2 : 1;
  float a = 0.f, b = 0.f;
  for (int q0 = pad0; q0 < pad1; q0 += T) {
    __syncthreads();
    if (ty == 0) {
      int ii = q0 + tx - pad0;
      if (ii >= n) ii = n - 1;
      toks[tx] = c.D1[off + ii];
    }
    __syncthreads();
    // Xs[kk][m] = x[tok(q0+kk)][blockIdx.x*T + m]
    const int im = blockIdx.x * T + tx;
    Xs[ty][tx] = im < c.d ? x[(int64_t)toks[ty] * c.d + im] : 0.f;
    const int64_t row = (int64_t)(q0 + ty) * nb * c.h;
    As[ty][tx] = j < c.h ? dAB[row + j] : 0.f;
    if (swiglu) Bs[ty][tx] = j < c.h ? dAB[row + c.h + j] : 0.f;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < T; ++kk) {
      a = fmaf(Xs[kk][ty], As[kk][tx], a);
      if (swiglu) b = fmaf(Xs[kk][ty], Bs[kk][tx], b);
    }
  }
  if (i >= c.d || j >= c.h) return;
  const int64_t o = ((int64_t)e * c.d + i) * c.h + j;
  dW1[o] = a;
  if (swiglu) dW2[o] = b;
}

// dW3_e[j][col] = sum_q Hg[q][j] dY[tok q][col]
__global__ void dw3_kernel(Common c, const float* __restrict__ Hg, const float* __restrict__ dY,
                           float* __restrict__ dW3) {
  if (!c.shape_ok()) return;
  __shared__ float Hs[T][T + 1], Gs[T][T + 1];
  __shared__ int toks[T];
  const int e = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int j = blockIdx.x * T + ty, col = blockIdx.y * T + tx;
  const int pad0 = c.meta.pad_off[e], pad1 = c.meta.pad_off[e + 1];
  const int off = c.D2[e], n = c.D2[e + 1] - off;
  float acc = 0.f;
  for (int q0 = pad0; q0 < pad1; q0 += T) {
    __syncthreads();
    if (ty == 0) {
      int ii = q0 + tx - pad0;
      if (ii >= n) ii = n - 1;
      toks[tx] = c.D1[off + ii];
    }
    __syncthreads();
    const int jm = blockIdx.x * T + tx;
    Hs[ty][tx] = jm < c.h ? Hg[(int64_t)(q0 + ty) * c.h + jm] : 0.f;
    Gs[ty][tx] = col < c.d ? dY[(int64_t)toks[ty] * c.d + col] : 0.f;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < T; ++kk) acc = fmaf(Hs[kk][ty], Gs[kk][tx], acc);
  }
  if (j >= c.h || col >= c.d) return;
  dW3[((int64_t)e * c.h + j) * c.d + col] = acc;
}

Common make_common(const moeblaze_shape& s, const moeblaze_dispatch& disp, const float* gates) {
  Common c;
  c.D1 = disp.expert_token_indices;
  c.D2 = disp.expert_token_offsets;
  c.D3 = disp.token_expert_indices;
  c.gates = gates;
  c.meta = meta_view(disp.meta, s.E);
  c.L = s.L; c.d = s.d; c.h = s.h; c.E = s.E; c.K = s.K;
  return c;
}

}  // namespace

moeblaze_status simt_forward(const moeblaze_shape& s, const float* x, const float* gates,
                             const moeblaze_dispatch& disp, const float* W1, const float* W2, const float* W3,
                             float* y, float* saved, float* wsH, cudaStream_t st) {
  const bool swiglu = s.act == MOEBLAZE_SWIGLU;
  const int64_t LK = s.L * s.K;
  const int64_t rows = max_padded_rows(LK, s.E);
  MB_CUDA(cudaMemsetAsync(y, 0, sizeof(float) * s.L * s.d, st));
  if (s.L == 0) return MOEBLAZE_OK;
  Common c = make_common(s, disp, gates);
  float* A = saved;
  float* B = swiglu ? saved + rows * s.h : nullptr;
  dim3 blk(T, T);
  stage_event(0, st);
  up_kernel<<<dim3((unsigned)(rows / T), (s.h + T - 1) / T), blk, 0, st>>>(c, x, W1, W2, A, B, wsH, rows, swiglu);
  MB_CUDA(cudaGetLastError());
  count_launch();
  stage_event(1, st);
  down_kernel<<<dim3((unsigned)(rows / T), (s.d + T - 1) / T), blk, 0, st>>>(c, wsH, W3, y);
  MB_CUDA(cudaGetLastError());
  count_launch();
  stage_event(2, st);
  stage_event(3, st);
  return MOEBLAZE_OK;
}

moeblaze_status simt_backward(const moeblaze_shape& s, const float* dY, const float* x, const float* gates,
                              const moeblaze_dispatch& disp, const float* W1, const float* W2, const float* W3,
                              const float* saved, float* dX, float* dW1, float* dW2, float* dW3, float* dgates,
                              float* wsdAB, float* wsHg, cudaStream_t st) {
  const bool swiglu = s.act == MOEBLAZE_SWIGLU;
  const int64_t LK = s.L * s.K;
  const int64_t rows = max_padded_rows(LK, s.E);
  MB_CUDA(cudaMemsetAsync(dX, 0, sizeof(float) * s.L * s.d, st));
  Common c = make_common(s, disp, gates);
  const float* A = saved;
  const float* B = swiglu ? saved + rows * s.h : nullptr;
  dim3 blk(T, T);
  stage_event(0, st);
  if (s.L > 0) {
    dh_kernel<<<dim3((unsigned)(rows / T), (s.h + T - 1) / T), blk, 0, st>>>(c, dY, W3, A, B, wsdAB, wsHg, dgates, swiglu);
    MB_CUDA(cudaGetLastError());
    count_launch();
    stage_event(1, st);
    dx_kernel<<<dim3((unsigned)(rows / T), (s.d + T - 1) / T), blk, 0, st>>>(c, wsdAB, W1, W2, dX, swiglu);
    MB_CUDA(cudaGetLastError());
    count_launch();
  }
  stage_event(2, st);
  dw12_kernel<<<dim3((s.d + T - 1) / T, (s.h + T - 1) / T, s.E), blk, 0, st>>>(c, x, wsdAB, dW1, dW2, swiglu);
  MB_CUDA(cudaGetLastError());
  count_launch();
  stage_event(3, st);
  dw3_kernel<<<dim3((s.h + T - 1) / T, (s.d + T - 1) / T, s.E), blk, 0, st>>>(c, wsHg, dY, dW3);
  MB_CUDA(cudaGetLastError());
  count_launch();
  stage_event(4, st);
  stage_event(5, st);
  return MOEBLAZE_OK;
}

}  // namespace moeblaze
