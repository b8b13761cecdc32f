// Gather + weighted combine of the identity expert (y[t] = sum_k g[t,k] x[t]
// through the index structures), the data movement of MoEBlaze's forward
// gather and fused write-back with the expert MLP taken out (MoEBlaze,
// awesome-system-papers page, section "免物化 token dispatch", Forward and
// Backward; the backward is the same kernel on dY -> dX).
//
// Schedule: a persistent CTA per SM walks windows of 8 tokens (window w, w +
// gridDim.x, ...) and, inside a window, column chunks of its rows.
//   producer warp   For a window it reads the 8*K positions of the window's
//                   (token, slot) pairs from token_index_map, ranks them
//                   ascending (expert-major order, the order in which the
//                   grouped expert GEMM walks its rows) and looks each one up
//                   in expert_token_indices: routed row r of the window is
//                   token D1[pos_r].  For every column chunk it then copies
//                   each routed row's chunk, in that order, into a ring stage
//                   with one bulk TMA copy per row (cp.async.bulk, completion
//                   counted in bytes on the stage's mbarrier).  The next
//                   window's positions are fetched while the current one is
//                   copied.
//   8 consumer warps  Warp j owns token j of the window: per chunk it sums
//                   the staged rows of token j times their gates (packed
//                   fp32x2 FMAs, fp32 accumulation) and writes its output
//                   chunk once with 16-byte stores.
// Each routed row is fetched through expert_token_indices; the K fetches of a
// token's row fall in one window, so the repeats after the first are served
// by L2.  No atomics; the routed (L*K, d) buffer never exists.  Every
// mbarrier wait is bounded (globaltimer): on expiry the CTA records
// kErrTimeout, lets its copies in flight land (bounded) and returns.
#include <climits>

#include "common.cuh"

namespace moeblaze {
namespace {

constexpr int kWin = 8;                                // tokens per window (one consumer warp each)
constexpr int kConsumerWarps = kWin;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + the producer warp
constexpr int kStageBytes = 64 * 1024;                 // routed-row chunks of one window per stage
constexpr int kStages = 3;
constexpr uint64_t kTimeoutNs = 4000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;

// Per stage, written by the producer before the stage's full barrier
// completes: which staged rows (and gates) belong to each token of the window.
struct StageDesc {
  int32_t nslot[kWin];
  int16_t slot[kWin][kMaxK];
  float gate[kWin][kMaxK];
};
constexpr int kDescBytes = (sizeof(StageDesc) + 15) / 16 * 16;
constexpr size_t kSmemBytes = 128 + (size_t)kStages * kStageBytes + (size_t)kStages * kDescBytes + 2 * kStages * 8 + 16;

struct IdParams {
  const uint8_t* src;   // (L, row_bytes): x (forward) or dY (backward)
  uint8_t* dst;         // (L, row_bytes): y or dX
  const int32_t* D1;
  const int32_t* D4;
  const float* gates;
  const int32_t* hdr;
  int32_t* err;
  int64_t L, LK, nwin;
  int E, K;
  int row_bytes;        // d * element size (a multiple of 16)
  int cb;               // bytes of a row per column chunk (a multiple of 16)
  int nch;              // column chunks per row
};

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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of `parity` of `bar`: false on expiry (the CTA's
// abort flag and the device error word are set) or once another role of the
// CTA has given up (abort_s set).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_s, int32_t* err,
                                             uint64_t limit_ns = kTimeoutNs) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (abort_s && *abort_s) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        if (abort_s) *abort_s = 1;
        if (err) atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}
// one routed-row chunk, global -> shared, completion counted on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// The producer's view of one window: lane l holds routed rows i = l and
// i = l + 32 of the window (i = (token - t0) * K + slot) in unranked order.
struct WinRows {
  int32_t pos[2];   // position in expert_token_indices (-1: no such row)
  float g[2];
  int32_t rank[2];  // staged row: place in ascending position order (expert-major)
  int32_t tok[2];   // token - t0 by expert_token_indices (-1: not staged)
  int32_t m[2];     // place among the staged rows of the same token, by rank
  int32_t cnt;      // lanes < kWin: staged rows of token `lane`
  int32_t nvalid;   // staged rows of the window (same in every lane)
};

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) identity_combine_kernel(const __grid_constant__ IdParams p) {
  constexpr int V = Vec<T>::N;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  StageDesc* desc = reinterpret_cast<StageDesc*>(smem + (size_t)kStages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * kStageBytes + (size_t)kStages * kDescBytes);
  volatile int* abort_s = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // a dispatch built for another (L, E, K): record it and read none of its maps
  // (the same three header words in every thread: the CTA leaves together)
  if (!meta_matches(p.hdr, p.L, p.E, p.K)) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrShapeMismatch);
    return;
  }
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + kStages + s); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumerWarps);
    }
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int n = kWin * p.K;  // routed rows of a window
  const uint32_t stage0 = smem_u32(smem);

  if (warp == kConsumerWarps) {
    // ================================================================ producer
    // first half of a window's preparation: its positions and gates
    auto load_rows = [&](int64_t w, WinRows& R) {
      const int64_t t0 = w * kWin;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        R.pos[h] = -1;
        R.g[h] = 0.f;
        if (i < n && t0 + i / p.K < p.L) {
          const int32_t q = p.D4[t0 * p.K + i];
          if (q >= 0 && q < p.LK) {
            R.pos[h] = q;
            R.g[h] = p.gates[t0 * p.K + i];
          }
        }
      }
    };
    // second part: the gather index of each routed row (loads issued here,
    // used in rank_b) and its expert-major rank
    auto rank_a = [&](WinRows& R, int32_t* tt) {
      int32_t key[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        key[h] = R.pos[h] >= 0 ? R.pos[h] : INT_MAX;
        tt[h] = R.pos[h] >= 0 ? p.D1[R.pos[h]] : -1;  // expert_token_indices: the token of this routed row
        R.rank[h] = 0;
      }
      for (int j = 0; j < n; ++j) {
        const int32_t kj = __shfl_sync(0xffffffffu, j < 32 ? key[0] : key[1], j & 31);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = lane + 32 * h;
          R.rank[h] += (kj < key[h]) || (kj == key[h] && j < i);
        }
      }
    };
    // third part: rows whose token lies in the window are staged; the
    // per-token lists in rank order
    auto rank_b = [&](int64_t w, WinRows& R, const int32_t* tt) {
      const int64_t t0 = w * kWin;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        R.tok[h] = -1;
        if (R.pos[h] >= 0 && (int64_t)tt[h] >= t0 && (int64_t)tt[h] < t0 + kWin && (int64_t)tt[h] < p.L)
          R.tok[h] = (int32_t)(tt[h] - t0);
      }
      R.m[0] = R.m[1] = 0;
      R.cnt = 0;
      int nv = 0;
      for (int j = 0; j < n; ++j) {
        const int32_t tj = __shfl_sync(0xffffffffu, j < 32 ? R.tok[0] : R.tok[1], j & 31);
        const int32_t rj = __shfl_sync(0xffffffffu, j < 32 ? R.rank[0] : R.rank[1], j & 31);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (R.tok[h] >= 0 && tj == R.tok[h] && rj < R.rank[h]) ++R.m[h];
        R.cnt += (tj == lane);
        nv += (tj >= 0);
      }
      R.nvalid = nv;
    };

    int s = 0;
    uint32_t ph = 0;
    uint32_t armed = 0, armed_par = 0;  // stages with copies issued, and the parity they complete
    bool ok = true;
    WinRows cur, nxt;
    int32_t tt[2];
    int64_t w = blockIdx.x;
    if (w < p.nwin) {
      load_rows(w, cur);
      rank_a(cur, tt);
      rank_b(w, cur, tt);
    }
    // the next window is prepared in three parts spread over this window's
    // chunks, so the latency of its index loads hides behind the copies
    const int c_b = p.nch > 1 ? 1 : 0;
    for (; ok && w < p.nwin; w += gridDim.x) {
      const int64_t wn = w + gridDim.x;
      if (wn < p.nwin) load_rows(wn, nxt);  // lands while this window's chunks are issued
      const int64_t t0 = w * kWin;
      for (int c = 0; c < p.nch; ++c) {
        bool got = true;
        if (lane == 0) got = wait_bounded(empty(s), ph ^ 1u, abort_s, p.err);
        ok = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        if (!ok) break;
        const int bytes = min(p.cb, p.row_bytes - c * p.cb);
        StageDesc& D = desc[s];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (cur.tok[h] >= 0 && cur.m[h] < kMaxK) {
            D.slot[cur.tok[h]][cur.m[h]] = (int16_t)cur.rank[h];
            D.gate[cur.tok[h]][cur.m[h]] = cur.g[h];
          }
        if (lane < kWin) D.nslot[lane] = min(cur.cnt, kMaxK);
        __syncwarp();  // the descriptor writes come before lane 0's arrive (release)
        if (lane == 0) mbar_arrive_expect_tx(full(s), (uint32_t)(cur.nvalid * bytes));
        __syncwarp();
        const uint32_t dst = stage0 + (uint32_t)s * kStageBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (cur.tok[h] >= 0)
            bulk_g2s(dst + (uint32_t)(cur.rank[h] * p.cb), p.src + (t0 + cur.tok[h]) * p.row_bytes + (int64_t)c * p.cb,
                     (uint32_t)bytes, full(s));
        armed |= 1u << s;
        armed_par = (armed_par & ~(1u << s)) | (ph << s);
        if (++s == kStages) { s = 0; ph ^= 1u; }
        if (c == 0 && wn < p.nwin) rank_a(nxt, tt);
        if (c == c_b && wn < p.nwin) rank_b(wn, nxt, tt);
      }
      if (ok && wn < p.nwin) cur = nxt;
    }
    if (!ok) {
      // let the copies already issued land before the CTA's shared memory goes away
      if (lane == 0)
        for (int i = 0; i < kStages; ++i)
          if (armed & (1u << i)) wait_bounded(full(i), (armed_par >> i) & 1u, nullptr, nullptr, kDrainNs);
      __syncwarp();
    }
  } else {
    // ================================================================ consumers
    const int j = warp;  // token j of each window
    int s = 0;
    uint32_t ph = 0;
    for (int64_t w = blockIdx.x; w < p.nwin; w += gridDim.x) {
      const int64_t t = w * kWin + j;
      bool ok = true;
      for (int c = 0; c < p.nch; ++c) {
        bool got = true;
        if (lane == 0) got = wait_bounded(full(s), ph, abort_s, p.err);
        ok = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        if (!ok) break;
        const int bytes = min(p.cb, p.row_bytes - c * p.cb);
        if (t < p.L) {
          const StageDesc& D = desc[s];
          const int ns = D.nslot[j];
          uint32_t base[kMaxK];
          float2 g2[kMaxK];
#pragma unroll
          for (int m = 0; m < kMaxK; ++m) {
            base[m] = (uint32_t)D.slot[j][m] * p.cb;
            g2[m] = make_float2(D.gate[j][m], D.gate[j][m]);
          }
          const uint8_t* stg = smem + (size_t)s * kStageBytes;
          uint8_t* out = p.dst + t * p.row_bytes + (int64_t)c * p.cb;
          for (int q = lane * 16; q < bytes; q += 32 * 16) {
            float2 acc[V / 2];
#pragma unroll
            for (int i = 0; i < V / 2; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int m = 0; m < kMaxK; ++m)
              if (m < ns) Vec<T>::fma(*reinterpret_cast<const uint4*>(stg + base[m] + q), g2[m], acc);
            *reinterpret_cast<uint4*>(out + q) = Vec<T>::pack(acc);
          }
        }
        __syncwarp();  // every lane has read the stage
        if (lane == 0) mbar_arrive(empty(s));
        if (++s == kStages) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
    }
  }
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
  const MetaView meta = meta_view(disp.meta, s.E);
  IdParams p;
  p.src = reinterpret_cast<const uint8_t*>(src);
  p.dst = reinterpret_cast<uint8_t*>(dst);
  p.D1 = disp.expert_token_indices;
  p.D4 = disp.token_index_map;
  p.gates = gates;
  p.hdr = meta.hdr;
  p.err = meta.err;
  p.L = s.L;
  p.LK = s.L * s.K;
  p.nwin = (s.L + kWin - 1) / kWin;
  p.E = s.E;
  p.K = s.K;
  p.row_bytes = s.d * (s.dtype == MOEBLAZE_BF16 ? 2 : 4);  // a multiple of 16 (checked by the ABI)
  // a stage holds one column chunk of the window's 8*K routed rows
  const int n = kWin * s.K;
  p.cb = (kStageBytes / n) / 16 * 16;
  if (p.cb > p.row_bytes) p.cb = p.row_bytes;
  p.nch = (p.row_bytes + p.cb - 1) / p.cb;
  const int64_t g64 = p.nwin < sm_count() ? p.nwin : sm_count();
  const dim3 grid((unsigned)g64);
  if (s.dtype == MOEBLAZE_BF16) {
    auto k = identity_combine_kernel<__nv_bfloat16>;
    MB_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
    k<<<grid, kThreads, kSmemBytes, st>>>(p);
  } else {
    auto k = identity_combine_kernel<float>;
    MB_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
    k<<<grid, kThreads, kSmemBytes, st>>>(p);
  }
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

}  // namespace moeblaze
