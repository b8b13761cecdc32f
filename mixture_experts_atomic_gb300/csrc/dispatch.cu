// Atomic-free three-step dispatch build (MoEBlaze, awesome-system-papers
// page, section "Atomic-free 三步 dispatch 构建").
//
//   K1 bitmap_kernel   one CTA per chunk of 1024 tokens (CTA 0 also clears
//                      the device error word).  Builds the chunk's
//                      token-expert bitmap in shared memory (bit t%32 of word
//                      [e][t/32]; every (t,e) bit written once: the lanes of a
//                      warp with the same expert are found by bit-plane
//                      ballots and only the lowest one writes, so no two
//                      lanes touch one word).  While the bitmap is on chip it
//                      derives, per expert, the prefix of set bits before
//                      every word (a shuffle scan over the expert's 32
//                      popcounts), the per (expert, chunk) count, and the
//                      in-chunk rank of every (token, slot):
//                      wordprefix + popc(bits below).  It writes the counts
//                      and the ranks (u16, token-major); the bitmap itself
//                      never goes to HBM.
//   K2 scan_kernel     one CTA per expert: the exclusive scan of its chunk
//                      counts -> chunk bases and n_e.  Large layers only:
//                      below chunks x experts = 32768 each K3 CTA sums the
//                      counts it needs itself (one launch fewer).
//   K3 scatter_kernel  one CTA per chunk, streaming: expert_token_offsets
//                      from a block scan of n_e; every (token, slot) gets
//                      pos = off[e] + base[e][c] + rank.  Writes
//                      token_index_map token-major (one vector per token);
//                      the chunk's tokens are staged in shared memory in
//                      expert_token_indices order, so each expert's run of
//                      that array is written by consecutive threads.
//                      The CTAs also split the GEMM metadata: padded row
//                      offsets, the tile -> expert table, the experts'
//                      descending-load order and the (L, E, K) the build was
//                      made for.
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

// dispatch workspace: (in-chunk rank << 16 | expert) [L][K] i32 | cnt/base [E][C] i32
struct DispatchWs {
  int32_t* packed;
  int32_t* base;
};

DispatchWs carve(void* ws, const moeblaze_shape& s) {
  DispatchWs w;
  w.packed = reinterpret_cast<int32_t*>(ws);
  const size_t rb = align_up((size_t)s.L * s.K * sizeof(int32_t), 256);
  w.base = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + rb);
  return w;
}

// Programmatic dependent launch: K2 and K3 are launched while the kernel
// before them is still running (its last CTAs have started), so their launch
// and CTA start-up overlap its tail; each waits for the previous kernel's
// completion and memory before it reads anything that kernel wrote.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_previous() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

constexpr int kThreads = 256;                       // 8 warps; warp w owns words w, w+8, w+16, w+24
constexpr int kPasses = kChunkTokens / kThreads;    // tokens per thread (4)
constexpr int kRow = kChunkWords + 1;               // padded shared row: conflict-free column walks
constexpr int kMaxIdBits = 9;                       // bits of an expert id below kMaxE
static_assert(kMaxE <= (1 << kMaxIdBits), "expert ids must fit in kMaxIdBits bits");

// The K int32 values of token t's row (-1 for slots past K or tokens past
// L); KM >= K.  Rows are 4K bytes, so K = 4 and K = 2 rows are one vector.
template <int KM>
__device__ __forceinline__ void load_slots(const int32_t* __restrict__ src0, int64_t t, int64_t L, int K, int* v) {
#pragma unroll
  for (int k = 0; k < KM; ++k) v[k] = -1;
  if (t >= L) return;
  const int32_t* src = src0 + t * K;
  if constexpr (KM == 4) {
    if (K == 4) {
      const int4 u = *reinterpret_cast<const int4*>(src);
      v[0] = u.x, v[1] = u.y, v[2] = u.z, v[3] = u.w;
      return;
    }
  }
  if (K == 2) {
    const int2 u = *reinterpret_cast<const int2*>(src);
    v[0] = u.x, v[1] = u.y;
  } else {
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (k < K) v[k] = src[k];
  }
}

template <int KM>
__device__ __forceinline__ void store_slots(int32_t* __restrict__ dst0, int64_t t, int K, const int* v) {
  int32_t* dst = dst0 + t * K;
  if constexpr (KM == 4) {
    if (K == 4) {
      *reinterpret_cast<int4*>(dst) = make_int4(v[0], v[1], v[2], v[3]);
      return;
    }
  }
  if (K == 2) {
    *reinterpret_cast<int2*>(dst) = make_int2(v[0], v[1]);
  } else {
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (k < K) dst[k] = v[k];
  }
}

// K1: one CTA per chunk of 1024 tokens.  All ids are loaded up front and
// copied to token_expert_indices; the chunk's bitmap is built in shared
// memory (word [e][w] holds the tokens 32w..32w+31 of the chunk routed to
// e); the per-(expert, chunk) popcounts are written expert-major for the
// scan, and every (token, slot) gets (in-chunk rank << 16 | expert),
// token-major, for the scatter (-1 for an id out of [0, E)).
template <int KM>
__global__ void __launch_bounds__(kThreads) bitmap_kernel(const int32_t* __restrict__ ids, int64_t L, int E, int K,
                                                          int32_t* __restrict__ D3, int32_t* __restrict__ packed,
                                                          int32_t* __restrict__ cnt, int64_t C, int32_t* err) {
  extern __shared__ uint32_t words[];  // [E][kRow]: a padded row keeps [e][w] and [e'][w] in different banks
  uint16_t* wpre = reinterpret_cast<uint16_t*>(words + E * kRow);  // [E][kRow]: set bits before word w
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  allow_dependents();  // K2 / K3 may start their CTAs once every K1 CTA has started
  const int64_t chunk = blockIdx.x;
  const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;  // bits of the largest expert id

  int e_k[kPasses][KM];
#pragma unroll
  for (int j = 0; j < kPasses; ++j) load_slots<KM>(ids, chunk * kChunkTokens + (warp + 8 * j) * 32 + lane, L, K, e_k[j]);
  // token_expert_indices is the ids as given
#pragma unroll
  for (int j = 0; j < kPasses; ++j) {
    const int64_t t = chunk * kChunkTokens + (warp + 8 * j) * 32 + lane;
    if (t < L) store_slots<KM>(D3, t, K, e_k[j]);
  }
  {
    const int nw = E * kRow;  // cleared 4 words at a time, then the 0-3 left over
    for (int i = tid; i < nw / 4; i += kThreads) reinterpret_cast<uint4*>(words)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < (nw & 3)) words[(nw & ~3) + tid] = 0u;
  }
  // A new build starts with a clean device error word; K3, which runs after
  // every K1 CTA has finished, records invalid routing in it.
  if (chunk == 0 && tid == 0) *err = 0;
  // ids out of [0, E) are left out of the bitmap (K3 reports them)
#pragma unroll
  for (int j = 0; j < kPasses; ++j)
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (e_k[j][k] >= E) e_k[j][k] = -1;
  __syncthreads();

  // Word [e][w] collects the lanes of this warp routed to e.  Within one
  // slot k each lane finds the lanes that share its expert: one ballot per
  // bit of the id, keeping the lanes whose bit agrees with its own (and a
  // first ballot dropping lanes with no valid id).  This is the mask
  // match_any would give, from ballots, which cost less to issue.  Only the
  // group's lowest lane writes; distinct groups write distinct words.  The
  // kPasses token groups of one slot write different words, so they run
  // without ordering between them; two slots may write the same word, so a
  // warp barrier separates the slots.
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    if (k >= K) break;  // K is the same for every lane
#pragma unroll
    for (int j = 0; j < kPasses; ++j) {
      const int w = warp + 8 * j;
      const int e = e_k[j][k];
      unsigned grp = __ballot_sync(0xffffffffu, e >= 0);
      const unsigned ue = (unsigned)e;
#pragma unroll
      for (int b = 0; b < kMaxIdBits; ++b) {
        if (b >= nbits) break;  // the same in every lane
        const unsigned bit = (ue >> b) & 1u;
        const unsigned plane = __ballot_sync(0xffffffffu, bit != 0u);
        grp &= plane ^ (bit - 1u);  // the plane where the bit is set, its complement where it is not
      }
      if (e >= 0 && lane == __ffs(grp) - 1) words[e * kRow + w] |= grp;
    }
    __syncwarp();
  }
  __syncthreads();

  // Word prefixes and the per-(expert, chunk) count (counts stored [E][C]
  // for the scan).
  if (E * 8 <= 2 * kThreads) {
    // few experts: thread i covers words 4g..4g+3 of expert i/8 (g = i%8);
    // the 8 threads of an expert are consecutive lanes and scan their
    // popcounts with shuffles
    for (int i0 = 0; i0 < E * 8; i0 += kThreads) {
      const int i = i0 + tid;
      const bool v = i < E * 8;
      const int e = i >> 3, g = i & 7;
      int c[4] = {0, 0, 0, 0};
      if (v) {
#pragma unroll
        for (int q = 0; q < 4; ++q) c[q] = __popc(words[e * kRow + 4 * g + q]);
      }
      const int mine = c[0] + c[1] + c[2] + c[3];
      int incl = mine;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if ((lane & 7) >= o) incl += u;
      }
      if (v) {
        int r = incl - mine;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          wpre[e * kRow + 4 * g + q] = (uint16_t)r;
          r += c[q];
        }
        if (g == 7) cnt[(int64_t)e * C + chunk] = incl;
      }
    }
  } else {
    // many experts: a thread walks one expert's 32 words (the padded rows
    // put the threads of a warp in different banks) with a running popcount
    for (int e = tid; e < E; e += kThreads) {
      const uint32_t* row = words + e * kRow;
      uint16_t* prow = wpre + e * kRow;
      int run = 0;
#pragma unroll
      for (int w = 0; w < kChunkWords; ++w) {
        prow[w] = (uint16_t)run;
        run += __popc(row[w]);
      }
      cnt[(int64_t)e * C + chunk] = run;
    }
  }
  __syncthreads();

  // (in-chunk rank << 16 | expert) of every (token, slot): the rank counts
  // the set bits of its expert before its own
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kPasses; ++j) {
    const int w = warp + 8 * j;
    const int64_t t = chunk * kChunkTokens + w * 32 + lane;
    if (t >= L) continue;
    int pk[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      const int e = e_k[j][k];
      pk[k] = -1;
      if (k < K && e >= 0) {
        const uint32_t r = (uint32_t)wpre[e * kRow + w] + (uint32_t)__popc(words[e * kRow + w] & below);
        pk[k] = (int)((r << 16) | (uint32_t)e);
      }
    }
    store_slots<KM>(packed, t, K, pk);
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

// Exclusive scan of kThreads values (one per thread) across the block.
__device__ __forceinline__ int block_excl_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v, lane);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < kThreads / 32 ? wsum[lane] : 0;
    const int xi = warp_incl_scan(x, lane);
    if (lane < kThreads / 32) wsum[lane] = xi - x;
    if (lane == kThreads / 32 - 1) *total = xi;
  }
  __syncthreads();
  const int r = incl - v + wsum[warp];
  __syncthreads();
  return r;
}

constexpr int kMaxScanVec = 4;  // K2: counts a thread keeps in registers, in 4-wide vectors

// K2: one CTA per expert: exclusive scan of its chunk counts (in place) and
// its total n_e.  Each thread sums a contiguous run of chunks.
__global__ void __launch_bounds__(kThreads) scan_kernel(int32_t* __restrict__ cnt, int64_t C, int32_t* __restrict__ n_e) {
  __shared__ int wsum[32];
  __shared__ int total;
  allow_dependents();
  wait_previous();  // K1's counts
  const int e = blockIdx.x;
  int32_t* row = cnt + (int64_t)e * C;
  const int64_t per = (C + kThreads - 1) / kThreads;
  const int64_t c0 = threadIdx.x * per, c1 = (c0 + per < C) ? c0 + per : C;
  if (C % 4 == 0 && per % 4 == 0 && per <= 4 * kMaxScanVec) {  // the same in every thread
    // 16-byte aligned runs (every row starts at e*C, a multiple of 4): one
    // vector load and one vector store per 4 counts, kept in registers
    int4 v[kMaxScanVec];
    int s = 0;
#pragma unroll
    for (int q = 0; q < kMaxScanVec; ++q) {
      const int64_t c = c0 + 4 * q;
      v[q] = (4 * q < per && c < c1) ? *reinterpret_cast<const int4*>(row + c) : make_int4(0, 0, 0, 0);
      s += v[q].x + v[q].y + v[q].z + v[q].w;
    }
    int run = block_excl_scan(s, wsum, &total);
#pragma unroll
    for (int q = 0; q < kMaxScanVec; ++q) {
      const int64_t c = c0 + 4 * q;
      if (4 * q < per && c < c1) {
        int4 o;
        o.x = run; run += v[q].x;
        o.y = run; run += v[q].y;
        o.z = run; run += v[q].z;
        o.w = run; run += v[q].w;
        *reinterpret_cast<int4*>(row + c) = o;
      }
    }
    if (threadIdx.x == 0) n_e[e] = total;
    return;
  }
  int s = 0;
  for (int64_t c = c0; c < c1; ++c) s += row[c];
  int run = block_excl_scan(s, wsum, &total);
  for (int64_t c = c0; c < c1; ++c) {
    const int v = row[c];
    row[c] = run;
    run += v;
  }
  if (threadIdx.x == 0) n_e[e] = total;
}

// K3: one CTA per chunk, streaming.  Every global read (the chunk's counts
// or bases, the packed (rank, expert) slots) is issued first.  Each CTA then
// derives the expert offsets itself: the per-expert totals n_e come from K2,
// or, for a small layer without K2 (chunks x experts <= kInlineBaseCounts),
// from summing the count array, which also gives this chunk's bases; a block
// scan of n_e (and of the padded counts and of this chunk's counts, in the
// same pass) gives expert_token_offsets, the padded offsets and the chunk's
// staging offsets.  Each (token, slot) then gets
// pos = off[e] + base[e][c] + rank; token_index_map is written token-major,
// one vector per token, and expert_token_indices[pos] = token.
// The GEMM metadata is split over the CTAs here: a slice of the tile ->
// expert table (binary search in the padded offsets), a slice of the experts'
// load ranks, and, in CTA 0, expert_token_offsets, the padded offsets, the
// counts, the tile count and the (L, E, K) the build was made for.
constexpr int kInlineBaseCounts = 32768;
constexpr int kT3 = 256;                      // K3 threads: four tokens each
constexpr int kP3 = kChunkTokens / kT3;

template <int KM>
__global__ void __launch_bounds__(kT3, KM <= 4 ? 5 : 1) scatter_kernel(int64_t L, int E, int K, const int32_t* __restrict__ packed,
                                                           int64_t C, const int32_t* __restrict__ cb, bool scanned,
                                                           const int32_t* __restrict__ n_e_in,
                                                           int32_t* __restrict__ D1, int32_t* __restrict__ D2,
                                                           int32_t* __restrict__ D4, MetaView meta, int64_t max_tiles) {
  extern __shared__ int32_t sm[];
  int32_t* off = sm;               // [E+1]: expert_token_offsets
  int32_t* poff = off + E + 1;     // [E+1]: padded row offsets
  int32_t* ne = poff + E + 1;      // [E]: tokens per expert
  int32_t* cbase = ne + E;         // [E]: this chunk's base in each expert
  int32_t* ccnt = cbase + E;       // [E]: this chunk's tokens in each expert
  int32_t* ebase = ccnt + E;       // [E]: off[e] + cbase[e], the expert's first position from this chunk
  int32_t* delta = ebase + E;      // [E]: ebase[e] - (the expert's first entry in the chunk's staging)
  int32_t* stage_t = delta + E;    // [kChunkTokens * KM]: the chunk's tokens in expert_token_indices order
  uint16_t* stage_e = reinterpret_cast<uint16_t*>(stage_t + kChunkTokens * KM);  // their experts
  __shared__ int nstage;
  __shared__ unsigned long long wtot[kT3 / 32];
  __shared__ int wctot[kT3 / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  wait_previous();  // K1's slots and counts, K2's bases
  const int64_t chunk = blockIdx.x;

  // ---- all global reads first
  if (scanned) {
    for (int e = tid; e < E; e += kT3) {
      const int n = n_e_in[e];
      const int b = cb[(int64_t)e * C + chunk];
      ne[e] = n;
      cbase[e] = b;
      ccnt[e] = (chunk + 1 < C ? cb[(int64_t)e * C + chunk + 1] : n) - b;
    }
  }
  int p_k[kP3][KM];
#pragma unroll
  for (int j = 0; j < kP3; ++j) load_slots<KM>(packed, chunk * kChunkTokens + tid + kT3 * j, L, K, p_k[j]);
  if (!scanned) {
    // small layer: a warp per expert sums its chunk counts, before this
    // chunk (the base) and over all chunks (n_e)
    for (int e = warp; e < E; e += kT3 / 32) {
      int before = 0, all = 0, mine = 0;
      for (int64_t c = lane; c < C; c += 32) {
        const int v = cb[(int64_t)e * C + c];
        all += v;
        if (c < chunk) before += v;
        if (c == chunk) mine = v;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        all += __shfl_xor_sync(0xffffffffu, all, o);
        mine += __shfl_xor_sync(0xffffffffu, mine, o);
      }
      if (lane == 0) {
        cbase[e] = before;
        ne[e] = all;
        ccnt[e] = mine;
      }
    }
  }
  __syncthreads();

  // ---- expert offsets (exclusive scan of n_e), padded offsets and the
  // chunk's staging offsets (scan of its own counts): thread i owns experts
  // [i*per, (i+1)*per); a warp scan, then the warps' totals.  n_e and its
  // padded value are packed in one 64-bit word (neither half's running sum
  // reaches 2^32).
  {
    const int per = (E + kT3 - 1) / kT3;
    const int e0 = tid * per;
    unsigned long long mine = 0ull;
    int cmine = 0;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const unsigned n = (unsigned)ne[e];
        mine += ((unsigned long long)((n + kRowPad - 1) / kRowPad * kRowPad) << 32) | n;
        cmine += ccnt[e];
      }
    }
    unsigned long long incl = mine;
    int cincl = cmine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xffffffffu, incl, o);
      const int cu = __shfl_up_sync(0xffffffffu, cincl, o);
      if (lane >= o) {
        incl += u;
        cincl += cu;
      }
    }
    if (lane == 31) {
      wtot[warp] = incl;
      wctot[warp] = cincl;
    }
    __syncthreads();
    unsigned long long run = incl - mine;
    int crun = cincl - cmine;
    for (int w2 = 0; w2 < warp; ++w2) {
      run += wtot[w2];
      crun += wctot[w2];
    }
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const int o0 = (int32_t)(run & 0xffffffffull);
        off[e] = o0;
        poff[e] = (int32_t)(run >> 32);
        ebase[e] = o0 + cbase[e];
        delta[e] = o0 + cbase[e] - crun;
        const unsigned n = (unsigned)ne[e];
        run += ((unsigned long long)((n + kRowPad - 1) / kRowPad * kRowPad) << 32) | n;
        crun += ccnt[e];
      }
    }
    if (tid == kT3 - 1) {
      off[E] = (int32_t)(run & 0xffffffffull);
      poff[E] = (int32_t)(run >> 32);
      nstage = crun;
    }
  }
  __syncthreads();  // publishes the offsets and nstage
  // Routing check, one comparison per chunk: with every id in [0, E) and no
  // id repeated within a token, the chunk's bitmap holds one bit per slot,
  // so its counts add up to tokens x K; an id out of range (K1 left it out)
  // or a repeated one (two slots, one bit) leaves the sum short.  One atomic
  // per CTA, and only for invalid routing.
  const int64_t ntok = min((int64_t)kChunkTokens, L - chunk * kChunkTokens);
  const bool any_bad = (int64_t)nstage != ntok * K;
  if (any_bad && tid == 0) atomicOr(meta.err, kErrBadRouting);

  // ---- place every (token, slot): token_index_map directly, the token into
  // the chunk's staging at its position minus delta[e] (the chunk's slots of
  // one expert are consecutive there, as in expert_token_indices)
#pragma unroll
  for (int j = 0; j < kP3; ++j) {
    const int64_t t = chunk * kChunkTokens + tid + kT3 * j;
    if (t >= L) continue;
    int d4[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      d4[k] = -1;
      if (k < K && p_k[j][k] >= 0) {
        const int e = p_k[j][k] & 0xffff;
        if (e < E) {
          const int pos = ebase[e] + (p_k[j][k] >> 16);
          const int si = pos - delta[e];
          stage_t[si] = (int32_t)t;
          stage_e[si] = (uint16_t)e;
          d4[k] = pos;
        }
      }
    }
    store_slots<KM>(D4, t, K, d4);
  }
  __syncthreads();
  // expert_token_indices: the chunk's runs, one per expert, each contiguous
  // in the output, written by consecutive threads.  A token with a repeated
  // id leaves a staging entry unwritten, so a chunk with invalid routing
  // skips this (its part of the output is unspecified; nothing is written
  // outside the buffer).
  if (!any_bad)
    for (int j = tid; j < nstage; j += kT3) D1[delta[stage_e[j]] + j] = stage_t[j];

  // ---- GEMM metadata, split over the CTAs
  // tile -> expert: tile m belongs to the expert whose padded rows hold row
  // 128 m (non-empty segments only own rows); -1 past the last tile
  const int64_t ntiles = poff[E] / kTileM;
  const int64_t per = (max_tiles + gridDim.x - 1) / gridDim.x;
  const int64_t m0 = (int64_t)blockIdx.x * per, m1 = min(max_tiles, m0 + per);
  for (int64_t m = m0 + tid; m < m1; m += kT3) {
    int32_t v = -1;
    if (m < ntiles) {
      const int64_t row = m * kTileM;
      int lo = 0, hi = E - 1;  // last e with poff[e] <= row
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (poff[mid] <= row) lo = mid;
        else hi = mid - 1;
      }
      v = lo;
    }
    meta.tile_expert[m] = v;
  }
  // descending load, equal loads by index: the rank of expert e is the number
  // of experts j with n_j > n_e, or n_j == n_e and j < e.  One warp per expert,
  // the experts spread over the CTAs.
  const int nwarps = kT3 / 32;
  for (int e = blockIdx.x * nwarps + warp; e < E; e += gridDim.x * nwarps) {
    const int32_t me = ne[e];
    int rank = 0;
    for (int jx = lane; jx < E; jx += 32) {
      const int32_t nj = ne[jx];
      rank += (nj > me) || (nj == me && jx < e);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (lane == 0) meta.order[rank] = e;
  }
  if (blockIdx.x != 0) return;
  if (tid == 0) {
    *meta.num_m_tiles = (int32_t)ntiles;
    *meta.padded_rows = poff[E];
    // the shape this build was made for, checked by every forward/backward kernel
    meta.hdr[kHdrL] = (int32_t)L;
    meta.hdr[kHdrE] = E;
    meta.hdr[kHdrK] = K;
  }
  for (int e = tid; e <= E; e += kT3) {
    D2[e] = off[e];
    meta.pad_off[e] = poff[e];
    if (e < E) meta.n_e[e] = ne[e];
  }
}

}  // namespace

namespace {

// Launch `kern` on `st` as a programmatic dependent of the kernel before it
// (the kernel calls wait_previous() before reading that kernel's output).
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}

// K2 (large layers) and K3 for ids of at most KM slots per token, once K1
// (or the router kernel that does K1's work) has written the packed slots
// and the per-(expert, chunk) counts.
template <int KM>
moeblaze_status run_tail(const moeblaze_shape& s, const moeblaze_dispatch& out, const DispatchWs& w,
                         const MetaView& meta, int64_t C, int64_t mt, cudaStream_t st) {
  const int E = s.E, K = s.K;
  const int64_t L = s.L;
  // Large layers scan each expert's chunk counts in K2 (one CTA per expert);
  // small ones let every K3 CTA sum the counts it needs.
  const bool scanned = C * E > kInlineBaseCounts;
  if (scanned) {
    MB_CUDA(launch_dependent(scan_kernel, dim3(E), dim3(kThreads), 0, st, w.base, C, meta.n_e));
    MB_CUDA(cudaGetLastError());
    count_launch();
  }
  const size_t sm3 = (size_t)(7 * E + 2) * sizeof(int32_t) + (size_t)kChunkTokens * KM * (sizeof(int32_t) + sizeof(uint16_t));
  if (sm3 > 48 * 1024)
    MB_CUDA(cudaFuncSetAttribute(scatter_kernel<KM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3));
  MB_CUDA(launch_dependent(scatter_kernel<KM>, dim3((unsigned)C), dim3(kT3), sm3, st, L, E, K, (const int32_t*)w.packed,
                           C, (const int32_t*)w.base, scanned, (const int32_t*)meta.n_e, out.expert_token_indices,
                           out.expert_token_offsets, out.token_index_map, meta, mt));
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

// K1, then the tail
template <int KM>
moeblaze_status run_build(const moeblaze_shape& s, const int32_t* ids, const moeblaze_dispatch& out,
                          const DispatchWs& w, const MetaView& meta, int64_t C, int64_t mt, cudaStream_t st) {
  const int E = s.E, K = s.K;
  const int64_t L = s.L;
  const size_t sm1 = (size_t)E * kRow * (sizeof(uint32_t) + sizeof(uint16_t));
  if (sm1 > 48 * 1024)
    MB_CUDA(cudaFuncSetAttribute(bitmap_kernel<KM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
  bitmap_kernel<KM><<<(unsigned)C, kThreads, sm1, st>>>(ids, L, E, K, out.token_expert_indices, w.packed, w.base, C,
                                                        meta.err);
  MB_CUDA(cudaGetLastError());
  count_launch();
  return run_tail<KM>(s, out, w, meta, C, mt, st);
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
  const int64_t C = num_chunks(s.L);
  return align_up((size_t)s.L * s.K * sizeof(int32_t), 256) + align_up((size_t)C * s.E * sizeof(int32_t), 256) + 256;
}

moeblaze_status launch_dispatch(const moeblaze_shape& s, const int32_t* ids, const moeblaze_dispatch& out,
                                void* ws, cudaStream_t st) {
  const int E = s.E, K = s.K;
  const int64_t L = s.L, LK = L * K;
  MetaView meta = meta_view(out.meta, E);
  const int64_t C = num_chunks(L);
  const int64_t mt = max_m_tiles(LK, E);
  if (L == 0) {
    // the header (error word, tile count, L = E = K = 0) is cleared here;
    // with tokens, K1 clears the error word and K3 writes the rest
    MB_CUDA(cudaMemsetAsync(out.meta, 0, 8 * sizeof(int32_t), st));
    // no tokens: offsets and counts are zero, no tiles
    MB_CUDA(cudaMemsetAsync(out.expert_token_offsets, 0, sizeof(int32_t) * (E + 1), st));
    MB_CUDA(cudaMemsetAsync(meta.n_e, 0, sizeof(int32_t) * (E + (E + 1)), st));
    MB_CUDA(cudaMemsetAsync(meta.tile_expert, 0xff, sizeof(int32_t) * mt, st));
    // order: identity permutation is not needed when there are no tiles
    MB_CUDA(cudaMemsetAsync(meta.order, 0, sizeof(int32_t) * E, st));
    return MOEBLAZE_OK;
  }
  DispatchWs w = carve(ws, s);
  if (K <= 2) return run_build<2>(s, ids, out, w, meta, C, mt, st);
  if (K <= 4) return run_build<4>(s, ids, out, w, meta, C, mt, st);
  return run_build<kMaxK>(s, ids, out, w, meta, C, mt, st);
}

void dispatch_ws_parts(const moeblaze_shape& s, void* ws, int32_t** packed, int32_t** cnt) {
  const DispatchWs w = carve(ws, s);
  *packed = w.packed;
  *cnt = w.base;
}

moeblaze_status launch_dispatch_tail(const moeblaze_shape& s, const moeblaze_dispatch& out, void* ws, cudaStream_t st) {
  const int K = s.K;
  const MetaView meta = meta_view(out.meta, s.E);
  const int64_t C = num_chunks(s.L);
  const int64_t mt = max_m_tiles(s.L * K, s.E);
  const DispatchWs w = carve(ws, s);
  if (K <= 2) return run_tail<2>(s, out, w, meta, C, mt, st);
  if (K <= 4) return run_tail<4>(s, out, w, meta, C, mt, st);
  return run_tail<kMaxK>(s, out, w, meta, C, mt, st);
}

}  // namespace moeblaze
