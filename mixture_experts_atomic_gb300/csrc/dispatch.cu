// Atomic-free three-step dispatch build (MoEBlaze, awesome-system-papers
// page, section "Atomic-free 三步 dispatch 构建").
//
//   K1 bitmap_kernel   one CTA per chunk of 1024 tokens.  Builds the chunk's
//                      token-expert bitmap in shared memory (bit t%32 of word
//                      [e][t/32]; every (t,e) bit written once, lanes with the
//                      same expert elected by match_any so no two lanes touch
//                      one word), writes it transposed (expert-major, each
//                      expert's 32 words = one 128-byte line) and the per
//                      (chunk, expert) popcount.
//   K2 scan_kernel     per expert, the exclusive scan of the chunk counts over
//                      chunks (warp shuffles) -> chunk bases and n_e.
//   K3 scatter_kernel  one CTA per chunk.  Scans n_e over experts ->
//                      expert_token_offsets; a per-expert warp scan of the
//                      chunk's 32 popcounts gives every word its first
//                      position; each token then places its K slots:
//                      pos = off[e] + base[c][e] + wordprefix + popc(bits below).
//                      Writes token_index_map and token_expert_indices
//                      coalesced (token-major) and expert_token_indices[pos].
//                      CTA 0 also writes the padded row offsets, the GEMM tile
//                      table and the experts' descending-load order.
//
// No global atomics on the data path (the device error word is the only
// atomic, and only for invalid routing).
#include <mutex>

#include "common.cuh"

namespace moeblaze {

namespace {

// Fixed scratch for callers that cannot allocate (moeblaze_dispatch_build_static).
// In host code this name is only a host-side stand-in: the device address is
// looked up per device with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[MOEBLAZE_STATIC_SCRATCH_BYTES];

// dispatch workspace: bitmap [E][C*32] u32 | cnt/base [C][E] i32
struct DispatchWs {
  uint32_t* bitmap;
  int32_t* base;
};

DispatchWs carve(void* ws, const moeblaze_shape& s) {
  int64_t C = num_chunks(s.L);
  DispatchWs w;
  w.bitmap = reinterpret_cast<uint32_t*>(ws);
  size_t bm = align_up((size_t)s.E * C * kChunkWords * sizeof(uint32_t), 256);
  w.base = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + bm);
  return w;
}

__global__ void __launch_bounds__(1024) bitmap_kernel(const int32_t* __restrict__ ids, int64_t L, int E, int K,
                                                      uint32_t* __restrict__ bitmap, int32_t* __restrict__ cnt,
                                                      int64_t words_per_expert, int32_t* err) {
  extern __shared__ uint32_t words[];  // [E][32]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t chunk = blockIdx.x;
  for (int i = tid; i < E * kChunkWords; i += blockDim.x) words[i] = 0u;
  __syncthreads();

  const int64_t t = chunk * kChunkTokens + tid;
  int e_k[kMaxK];
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) {
    e_k[k] = -1;
    if (k < K && t < L) {
      int e = ids[t * K + k];
      if (e < 0 || e >= E) { bad = true; e = -1; }
      e_k[k] = e;
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxK; ++k)
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k && k < K && e_k[k] >= 0 && e_k[k] == e_k[j]) bad = true;
  if (bad) atomicOr(err, kErrBadRouting);

  // Word [e][warp] collects the lanes of this warp routed to e.  Within one
  // slot k the lanes sharing an expert are grouped by match_any and only the
  // group's lowest lane writes; distinct groups write distinct words.
  for (int k = 0; k < K; ++k) {
    const int e = e_k[k];
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(grp) - 1) words[e * kChunkWords + warp] |= grp;
    __syncwarp();
  }
  __syncthreads();

  // transposed store: expert e's 32 words of this chunk are one 128-byte line
  for (int i = tid; i < E * kChunkWords; i += blockDim.x) {
    const int e = i / kChunkWords, w = i % kChunkWords;
    bitmap[(int64_t)e * words_per_expert + chunk * kChunkWords + w] = words[i];
  }
  // per-(chunk, expert) popcount: warp per expert, shuffle reduction
  for (int e = warp; e < E; e += blockDim.x / 32) {
    int v = __popc(words[e * kChunkWords + lane]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) cnt[chunk * E + e] = v;
  }
}

// One CTA per 32 experts (lane = expert); the warps split the chunks, each
// sums its range, the per-warp sums are scanned in shared memory and a second
// pass writes the exclusive chunk bases in place of the counts.
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ cnt, int64_t C, int E,
                                                    int32_t* __restrict__ n_e) {
  __shared__ int32_t part[32][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int64_t per = (C + nw - 1) / nw;
  const int64_t c0 = warp * per, c1 = (c0 + per < C) ? c0 + per : C;
  int32_t s = 0;
  if (e < E)
    for (int64_t c = c0; c < c1; ++c) s += cnt[c * E + e];
  part[warp][lane] = s;
  __syncthreads();
  if (warp == 0) {
    int32_t run = 0;
    for (int w = 0; w < nw; ++w) {
      int32_t v = part[w][lane];
      part[w][lane] = run;
      run += v;
    }
    if (e < E) n_e[e] = run;
  }
  __syncthreads();
  int32_t run = part[warp][lane];
  if (e < E)
    for (int64_t c = c0; c < c1; ++c) {
      int32_t v = cnt[c * E + e];
      cnt[c * E + e] = run;
      run += v;
    }
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

__global__ void __launch_bounds__(1024) scatter_kernel(const int32_t* __restrict__ ids, int64_t L, int E, int K,
                                                       const uint32_t* __restrict__ bitmap, int64_t words_per_expert,
                                                       const int32_t* __restrict__ base, const int32_t* __restrict__ n_e,
                                                       int32_t* __restrict__ D1, int32_t* __restrict__ D2,
                                                       int32_t* __restrict__ D3, int32_t* __restrict__ D4,
                                                       MetaView meta, int64_t max_tiles) {
  extern __shared__ int32_t sm[];
  uint32_t* words = reinterpret_cast<uint32_t*>(sm);  // [E][32]
  int32_t* wpre = sm + E * kChunkWords;               // [E][32]
  int32_t* off = wpre + E * kChunkWords;              // [E+1], then the chunk bases [E]
  __shared__ int32_t wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int64_t chunk = blockIdx.x;

  // exclusive scan of n_e over experts (E <= 1024 = blockDim)
  int v = (tid < E) ? n_e[tid] : 0;
  int incl = warp_incl_scan(v, lane);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < nw) ? wsum[lane] : 0;
    wsum[lane] = warp_incl_scan(w, lane) - w;
  }
  __syncthreads();
  if (tid < E) off[tid] = incl - v + wsum[warp];
  if (tid == E - 1) off[E] = incl + wsum[warp];
  for (int i = tid; i < E * kChunkWords; i += blockDim.x) {
    const int e = i / kChunkWords, w = i % kChunkWords;
    words[i] = bitmap[(int64_t)e * words_per_expert + chunk * kChunkWords + w];
  }
  // the chunk's per-expert bases, staged with the words (one coalesced read)
  int32_t* cbase = off + E + 1;
  if (tid < E) cbase[tid] = base[chunk * E + tid];
  __syncthreads();

  // first position of every (expert, word): warp per expert
  for (int e = warp; e < E; e += nw) {
    const int c = __popc(words[e * kChunkWords + lane]);
    const int in = warp_incl_scan(c, lane);
    wpre[e * kChunkWords + lane] = off[e] + cbase[e] + in - c;
  }
  __syncthreads();

  const int64_t t = chunk * kChunkTokens + tid;
  if (t < L) {
    const int w = tid >> 5, b = tid & 31;
    const uint32_t below = (1u << b) - 1u;
    for (int k = 0; k < K; ++k) {
      const int e = ids[t * K + k];
      int32_t pos = -1;
      if (e >= 0 && e < E) {
        pos = wpre[e * kChunkWords + w] + __popc(words[e * kChunkWords + w] & below);
        D1[pos] = (int32_t)t;
      }
      D3[t * K + k] = e;
      D4[t * K + k] = pos;
    }
  }

  if (chunk == 0) {
    // offsets, padded offsets, tile table, load order (CTA 0 only)
    __shared__ int32_t poff[kMaxE + 1];
    for (int e = tid; e <= E; e += blockDim.x) D2[e] = off[e];
    if (tid == 0) {
      int32_t run = 0;
      for (int e = 0; e < E; ++e) {
        poff[e] = run;
        meta.pad_off[e] = run;
        int32_t n = off[e + 1] - off[e];
        run += (n + kRowPad - 1) / kRowPad * kRowPad;
      }
      poff[E] = run;
      meta.pad_off[E] = run;
      *meta.num_m_tiles = run / kTileM;
      *meta.padded_rows = run;
    }
    __syncthreads();
    const int32_t ntiles = poff[E] / kTileM;
    for (int64_t m = tid; m < max_tiles; m += blockDim.x) {
      int32_t ex = -1;
      if (m < ntiles) {  // binary search: last e with poff[e] <= m*128
        int lo = 0, hi = E - 1;
        const int32_t r = (int32_t)m * kTileM;
        while (lo < hi) {
          int mid = (lo + hi + 1) >> 1;
          if (poff[mid] <= r) lo = mid; else hi = mid - 1;
        }
        ex = lo;
      }
      meta.tile_expert[m] = ex;
    }
    if (tid < E) {
      const int32_t me = off[tid + 1] - off[tid];
      int rank = 0;
      for (int j = 0; j < E; ++j) {
        const int32_t nj = off[j + 1] - off[j];
        rank += (nj > me) || (nj == me && j < tid);
      }
      meta.order[rank] = tid;
    }
  }
}

}  // namespace

moeblaze_status launch_dispatch_static(const moeblaze_shape& s, const int32_t* ids, const moeblaze_dispatch& out,
                                       cudaStream_t st) {
  constexpr int kMaxDev = 64;
  static void* addr[kMaxDev] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  MB_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDev) return MOEBLAZE_ERR_UNSUPPORTED;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
      // one-time set-up on this device (the current one): the array's device address
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MOEBLAZE_ERR_CUDA;
      addr[dev] = p;
    }
    ws = addr[dev];
  }
  return launch_dispatch(s, ids, out, ws, st);
}

size_t dispatch_ws_bytes(const moeblaze_shape& s) {
  int64_t C = num_chunks(s.L);
  return align_up((size_t)s.E * C * kChunkWords * sizeof(uint32_t), 256) +
         align_up((size_t)C * s.E * sizeof(int32_t), 256) + 256;
}

moeblaze_status launch_dispatch(const moeblaze_shape& s, const int32_t* ids, const moeblaze_dispatch& out,
                                void* ws, cudaStream_t st) {
  const int E = s.E, K = s.K;
  const int64_t L = s.L, LK = L * K;
  MetaView meta = meta_view(out.meta, E);
  MB_CUDA(cudaMemsetAsync(out.meta, 0, 8 * sizeof(int32_t), st));
  const int64_t C = num_chunks(L);
  const int64_t mt = max_m_tiles(LK, E);
  if (L == 0) {
    // no tokens: offsets and counts are zero, no tiles
    MB_CUDA(cudaMemsetAsync(out.expert_token_offsets, 0, sizeof(int32_t) * (E + 1), st));
    MB_CUDA(cudaMemsetAsync(meta.n_e, 0, sizeof(int32_t) * (E + (E + 1)), st));
    MB_CUDA(cudaMemsetAsync(meta.tile_expert, 0xff, sizeof(int32_t) * mt, st));
    // order: identity permutation is not needed when there are no tiles
    MB_CUDA(cudaMemsetAsync(meta.order, 0, sizeof(int32_t) * E, st));
    return MOEBLAZE_OK;
  }
  DispatchWs w = carve(ws, s);
  const int64_t wpe = C * kChunkWords;
  size_t sm1 = (size_t)E * kChunkWords * sizeof(uint32_t);
  if (sm1 > 48 * 1024) MB_CUDA(cudaFuncSetAttribute(bitmap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
  bitmap_kernel<<<(unsigned)C, 1024, sm1, st>>>(ids, L, E, K, w.bitmap, w.base, wpe, meta.err);
  MB_CUDA(cudaGetLastError());
  count_launch();
  scan_kernel<<<(E + 31) / 32, 1024, 0, st>>>(w.base, C, E, meta.n_e);
  MB_CUDA(cudaGetLastError());
  count_launch();
  size_t sm3 = (size_t)E * kChunkWords * 8 + (2 * E + 1) * sizeof(int32_t);
  if (sm3 > 48 * 1024) MB_CUDA(cudaFuncSetAttribute(scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3));
  scatter_kernel<<<(unsigned)C, 1024, sm3, st>>>(ids, L, E, K, w.bitmap, wpe, w.base, meta.n_e,
                                                  out.expert_token_indices, out.expert_token_offsets,
                                                  out.token_expert_indices, out.token_index_map, meta, mt);
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

}  // namespace moeblaze
