// The softmax top-K router fused with the first step of the atomic-free
// dispatch (MoEBlaze, awesome-system-papers page: the token-choice top-K
// routing that produces the ids, and section "Atomic-free 三步 dispatch 构建"
// for the bitmap): one kernel computes the logits on the tensor cores, picks
// the K experts and their softmax gates, and, while the ids are still in
// registers, builds the chunk's token-expert bitmap on chip and emits what
// the dispatch's first kernel would (per-(expert, chunk) counts and every
// slot's in-chunk rank).  The ids never make a round trip through HBM before
// the bitmap exists.
//
// Logits on the tensor cores, at fp32 precision: Wr (fp32) is split into
// three bf16 parts, Wr = hi + mid + lo (each the bf16 rounding of what the
// parts before it leave), so that x . Wr = x . hi + x . mid + x . lo with
// every product exact and the sum accumulated in fp32 in TMEM.  The three
// parts are the rows of one B operand [hi | mid | lo] (EP rows each, EP the
// expert count rounded up to 8, 16, 32 or 64), so one MMA per 16-deep
// k-slice gives all three partial logits.
//
// Grid: one CTA per 128 tokens, clusters of 8 CTAs = one 1024-token dispatch
// chunk.  Warp 4 streams the CTA's x tile and the split weights by TMA
// through a 4-stage ring (2 stages for 64 experts), warp 5 allocates TMEM and issues
// tcgen05.mma.cta_group::1.kind::f16 (M = 128, N = 3 EP rounded up to 16),
// warps 0-3 (one token per thread, TMEM lanes 32w..32w+31) read the
// accumulator row, add the three parts and the bias, select the top K
// (larger first, equal logits to the lower index) and write ids, gates and
// token_expert_indices.  Each warp's 32 tokens then form one bitmap word per
// expert (a ballot per expert); the CTAs of the cluster exchange their
// per-expert popcounts through distributed shared memory, so each CTA knows
// how many of the chunk's earlier tokens every expert has, and every slot
// gets its in-chunk rank: earlier CTAs + earlier words of this CTA + the
// bits below it in its own word.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moeblaze {
namespace tc {
namespace {

constexpr int kRtTokens = 128;                      // tokens per CTA (one M tile)
constexpr int kRtThreads = 192;                     // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr int kRtCluster = kChunkTokens / kRtTokens;  // CTAs of one dispatch chunk (8)
constexpr int kRtA = kRtTokens * 64 * 2;            // one x k-block: 16 KB
constexpr int kRtMaxEP = 64;

__host__ __device__ constexpr int rt_n(int ep) { return (3 * ep + 15) / 16 * 16; }
__host__ __device__ constexpr int rt_cols(int ep) {
  return rt_n(ep) <= 32 ? 32 : rt_n(ep) <= 64 ? 64 : rt_n(ep) <= 128 ? 128 : 256;
}
__host__ __device__ constexpr int rt_stage(int ep) { return kRtA + rt_n(ep) * 128; }
// ring depth: 4 stages, 2 for 64 experts, whose 40 KB stages would otherwise
// leave room for one CTA per SM (a cluster of 8 then needs 8 free SMs of a GPC)
__host__ __device__ constexpr int rt_stages(int ep) { return ep >= 64 ? 2 : 4; }
// ring | barriers, TMEM address, abort flag | bitmap words [EP][4] | popcounts [EP] | bases [EP] | 1 KB alignment slack
__host__ __device__ constexpr int rt_smem(int ep) { return rt_stages(ep) * rt_stage(ep) + 256 + ep * 4 * 4 + 2 * ep * 4 + 1024; }

struct RtParams {
  CUtensorMap tmX;  // x (L x d bf16), boxes of 64 columns x 128 rows
  CUtensorMap tmW;  // split weights (N x d bf16), boxes of 64 columns x N rows
  const float* bias;
  int64_t L, C;
  int d, E, K, kblocks;
  int32_t* ids;
  float* gates;
  int32_t* D3;
  int32_t* packed;
  int32_t* cnt;
  int32_t* err;
  uint64_t wait_ns;
};

// Wr (d x E fp32, row-major) -> [hi | mid | lo] (N x d bf16, K-major rows;
// rows of experts >= E and rows past 3 EP are zero)
__global__ void split_weights_kernel(const float* __restrict__ Wr, int d, int E, int EP, int N,
                                     __nv_bfloat16* __restrict__ ws) {
  const int64_t n_all = (int64_t)N * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_all; i += (int64_t)gridDim.x * blockDim.x) {
    const int n = (int)(i / d), c = (int)(i % d);
    const int part = n / EP, e = n % EP;
    float v = 0.f;
    if (part < 3 && e < E) {
      const float w = Wr[(int64_t)c * E + e];
      const float hi = __bfloat162float(__float2bfloat16_rn(w));
      const float r1 = w - hi;  // exact
      const float mid = __bfloat162float(__float2bfloat16_rn(r1));
      v = part == 0 ? hi : part == 1 ? mid : r1 - mid;  // r1 - mid exact; rounded to bf16 below
    }
    ws[i] = __float2bfloat16_rn(v);
  }
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

template <int EP>
__global__ void __launch_bounds__(kRtThreads, 1) router_k1_kernel(const __grid_constant__ RtParams p) {
  constexpr int N = rt_n(EP), TCOLS = rt_cols(EP), SB = rt_stage(EP), kRtStages = rt_stages(EP);
  constexpr int NLD = (3 * EP + 31) / 32;  // 32-column TMEM loads that cover the three parts
  extern __shared__ uint8_t rt_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rt_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRtStages * SB);  // full[S], empty[S], done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kRtStages + 1);
  volatile int* abort_s = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* sw = reinterpret_cast<uint32_t*>(smem + kRtStages * SB + 256);  // [EP][4]: this CTA's words
  int* tot = reinterpret_cast<int*>(sw + EP * 4);                            // [EP]: their popcounts
  int* base = tot + EP;                                                       // [EP]: the chunk's earlier CTAs

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int64_t chunk = blockIdx.x / kRtCluster;
  const int64_t t0 = (int64_t)blockIdx.x * kRtTokens;
  const bool active = t0 < p.L;  // the same for the whole CTA
  const uint32_t smem_base = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + kRtStages + s); };
  const uint32_t done = smem_u32(bars + 2 * kRtStages);
  const uint64_t lim = p.wait_ns;

  // the dispatch's next kernels are launched as programmatic dependents: they
  // may start their CTAs once every CTA of this one has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0 && tid == 0) *p.err = 0;  // a new build starts with a clean error word
  if (tid == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (active && warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = active ? *tmem_slot : 0u;

  // per token (warps 0-3): the selected experts; the mask of them for the ballots
  int seli[kMaxK];
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) seli[k] = -1;
  const int64_t t = t0 + warp * 32 + lane;
  const bool valid = warp < 4 && t < p.L;

  if (active) {
    if (warp == 4) {
      // ============================================================ TMA producer
      if (lane == 0) {
        int s = 0;
        uint32_t ph = 0, armed = 0, armed_par = 0;
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!wait_bounded(empty(s), ph ^ 1u, abort_s, p.err, lim)) break;
          const uint32_t sA = smem_base + s * SB;
          mbar_expect_tx(full(s), (uint32_t)SB);
          tma_load_2d(sA, &p.tmX, kb * 64, (int)t0, full(s));
          tma_load_2d(sA + kRtA, &p.tmW, kb * 64, 0, full(s));
          armed |= 1u << s;
          armed_par = (armed_par & ~(1u << s)) | (ph << s);
          if (++s == kRtStages) { s = 0; ph ^= 1u; }
        }
        // a CTA that gave up lets its copies in flight land before it exits
        if (*abort_s)
          for (int i = 0; i < kRtStages; ++i)
            if ((armed >> i) & 1u) wait_bounded(full(i), (armed_par >> i) & 1u, nullptr, nullptr, kDrainNs);
      }
    } else if (warp == 5) {
      // ============================================================ MMA issuer
      if (lane == 0) {
        const uint32_t idesc = instr_desc(N, false, false);
        int s = 0;
        uint32_t ph = 0;
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!wait_bounded(full(s), ph, abort_s, p.err, lim)) break;
          tc_fence_after();
          const uint32_t sA = smem_base + s * SB, sB = sA + kRtA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem_base, smem_desc(sA + kk * 32, 16, 1024), smem_desc(sB + kk * 32, 16, 1024), idesc,
                     (kb | kk) ? 1u : 0u);
          mma_commit(empty(s));
          if (++s == kRtStages) { s = 0; ph ^= 1u; }
        }
        mma_commit(done);  // also after giving up: every MMA issued retires before TMEM is read or freed
        wait_bounded(done, 0u, nullptr, nullptr, *abort_s ? kDrainNs : lim);
      }
      __syncwarp();
    } else {
      // ============================================================ logits, top K, gates
      // warp-uniform: the TMEM loads below are warp-collective
      const bool ok = __all_sync(0xffffffffu, wait_bounded(done, 0u, abort_s, p.err, lim));
      tc_fence_after();
      float lg[EP];
#pragma unroll
      for (int e = 0; e < EP; ++e) lg[e] = 0.f;
      if (ok) {
#pragma unroll
        for (int q = 0; q < NLD; ++q) {
          uint32_t v[32];
          MB_TMEM_LD32(tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(q * 32), v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = q * 32 + i;
            if (c < 3 * EP) lg[c % EP] += __uint_as_float(v[i]);
          }
        }
      }
      if (valid) {
#pragma unroll
        for (int e = 0; e < EP; ++e) lg[e] = e < p.E ? lg[e] + (p.bias ? p.bias[e] : 0.f) : -FLT_MAX;
        unsigned long long taken = 0ull;
        float selv[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
          selv[k] = 0.f;
          if (k < p.K) {
            float bv = -FLT_MAX;
            int bi = INT_MAX;
#pragma unroll
            for (int e = 0; e < EP; ++e)
              if (!((taken >> e) & 1ull) && e < p.E && (lg[e] > bv || (lg[e] == bv && e < bi))) {
                bv = lg[e];
                bi = e;
              }
            selv[k] = bv;
            seli[k] = bi;
            taken |= 1ull << bi;
          }
        }
        float w[kMaxK], sum = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
          w[k] = k < p.K ? expf(selv[k] - selv[0]) : 0.f;
          sum += w[k];
        }
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
          if (k < p.K) {
            p.ids[t * p.K + k] = seli[k];
            p.D3[t * p.K + k] = seli[k];
            p.gates[t * p.K + k] = w[k] / sum;
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- bitmap
  // warp w (< 4) of this CTA covers the chunk's word 4 rank + w: one ballot
  // per expert; lane e % 32 keeps expert e's word
  if (warp < 4) {
    unsigned long long mine = 0ull;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k)
      if (valid && k < p.K) mine |= 1ull << seli[k];
    uint32_t wv[(EP + 31) / 32];
#pragma unroll
    for (int i = 0; i < (EP + 31) / 32; ++i) wv[i] = 0u;
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      const uint32_t m = __ballot_sync(0xffffffffu, (mine >> e) & 1ull);
      if (lane == (e & 31)) wv[e >> 5] = m;
    }
#pragma unroll
    for (int i = 0; i < (EP + 31) / 32; ++i)
      if (32 * i + lane < EP) sw[(32 * i + lane) * 4 + warp] = wv[i];
  }
  __syncthreads();
  if (tid < EP) tot[tid] = __popc(sw[tid * 4 + 0]) + __popc(sw[tid * 4 + 1]) + __popc(sw[tid * 4 + 2]) + __popc(sw[tid * 4 + 3]);
  cluster_sync();  // every CTA's popcounts are visible to the cluster
  if (tid < p.E) {
    const uint32_t a = smem_u32(tot + tid);
    int before = 0, all = 0;
    for (uint32_t r = 0; r < (uint32_t)kRtCluster; ++r) {
      const int v = ld_cluster_s32(peer_addr(a, r));
      all += v;
      if (r < rank) before += v;
    }
    base[tid] = before;
    if (rank == 0) p.cnt[(int64_t)tid * p.C + chunk] = all;
  }
  cluster_sync();  // no CTA reads another's popcounts after this; bases visible in the CTA

  // ---------------------------------------------------------------- ranks
  if (valid) {
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      if (k < p.K) {
        const int e = seli[k];
        int r = base[e] + __popc(sw[e * 4 + warp] & below);
#pragma unroll
        for (int w2 = 0; w2 < 3; ++w2)
          if (w2 < warp) r += __popc(sw[e * 4 + w2]);
        p.packed[t * p.K + k] = (r << 16) | e;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (active && warp == 5)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TCOLS) : "memory");
}

template <int EP>
moeblaze_status launch_ep(const moeblaze_shape& s, const void* x, const float* Wr, const float* bias, int32_t* ids,
                          float* gates, const moeblaze_dispatch& out, int32_t* packed, int32_t* cnt,
                          __nv_bfloat16* wsplit, cudaStream_t st) {
  constexpr int N = rt_n(EP);
  {
    const int64_t n = (int64_t)N * s.d;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4 * (int64_t)sm_count()) blocks = 4 * (int64_t)sm_count();
    split_weights_kernel<<<(unsigned)blocks, 256, 0, st>>>(Wr, s.d, s.E, EP, N, wsplit);
    MB_CUDA(cudaGetLastError());
    count_launch();
  }
  RtParams p;
  memset(&p, 0, sizeof(p));
  if (!make_map(&p.tmX, x, (uint64_t)s.d, (uint64_t)s.L, 64, kRtTokens)) return MOEBLAZE_ERR_CUDA;
  if (!make_map(&p.tmW, wsplit, (uint64_t)s.d, (uint64_t)N, 64, N)) return MOEBLAZE_ERR_CUDA;
  p.bias = bias;
  p.L = s.L;
  p.C = num_chunks(s.L);
  p.d = s.d;
  p.E = s.E;
  p.K = s.K;
  p.kblocks = s.d / 64;
  p.ids = ids;
  p.gates = gates;
  p.D3 = out.token_expert_indices;
  p.packed = packed;
  p.cnt = cnt;
  p.err = meta_view(out.meta, s.E).err;
  int withhold = 0;
  fault_injection(&p.wait_ns, &withhold);
  if (p.wait_ns == 0) p.wait_ns = kTimeoutNs;

  auto kern = router_k1_kernel<EP>;
  const int smem = rt_smem(EP);
  MB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRtCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(p.C * kRtCluster));
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  MB_CUDA(cudaLaunchKernelEx(&cfg, kern, p));
  count_launch();
  return MOEBLAZE_OK;
}

int padded_router_experts(int E) { return E <= 8 ? 8 : E <= 16 ? 16 : E <= 32 ? 32 : 64; }

}  // namespace
}  // namespace tc

size_t router_dispatch_ws_bytes(const moeblaze_shape& s) {
  const int EP = s.E <= tc::kRtMaxEP ? tc::padded_router_experts(s.E) : 0;
  return dispatch_ws_bytes(s) + align_up((size_t)tc::rt_n(EP) * s.d * sizeof(__nv_bfloat16), 256);
}

// the fused kernel takes bf16 x, up to 64 experts and at least one full
// 128-token tile (the x tile's TMA box)
bool router_dispatch_fused(const moeblaze_shape& s) {
  return s.dtype == MOEBLAZE_BF16 && s.E <= tc::kRtMaxEP && s.L >= tc::kRtTokens;
}

moeblaze_status launch_router_dispatch(const moeblaze_shape& s, const void* x, const float* Wr, const float* bias,
                                       int32_t* ids, float* gates, const moeblaze_dispatch& out, void* ws,
                                       cudaStream_t st) {
  int32_t* packed = nullptr;
  int32_t* cnt = nullptr;
  dispatch_ws_parts(s, ws, &packed, &cnt);
  auto* wsplit = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + dispatch_ws_bytes(s));
  moeblaze_status r = MOEBLAZE_OK;
  switch (tc::padded_router_experts(s.E)) {
    case 8: r = tc::launch_ep<8>(s, x, Wr, bias, ids, gates, out, packed, cnt, wsplit, st); break;
    case 16: r = tc::launch_ep<16>(s, x, Wr, bias, ids, gates, out, packed, cnt, wsplit, st); break;
    case 32: r = tc::launch_ep<32>(s, x, Wr, bias, ids, gates, out, packed, cnt, wsplit, st); break;
    default: r = tc::launch_ep<64>(s, x, Wr, bias, ids, gates, out, packed, cnt, wsplit, st); break;
  }
  if (r != MOEBLAZE_OK) return r;
  return launch_dispatch_tail(s, out, ws, st);
}

}  // namespace moeblaze
