// bf16 expert GEMMs of the layer on the sm_103a tensor cores (tcgen05 + TMEM,
// operands staged by TMA), with the index-driven row gather and the fused
// epilogues of MoEBlaze (awesome-system-papers page, sections
// "免物化 token dispatch" and "SwiGLU kernel 融合 + activation checkpoint").
//
// One persistent, warp-specialised kernel template serves all six GEMMs:
//   warps 0-3   producer: tiled TMA loads (thread 0) of the weight and
//               activation tiles into a 4-stage ring; the routed rows of x /
//               dY are gathered straight from the (L,d) tensor through
//               expert_token_indices by all 128 producer threads with 16-byte
//               cp.async into the 128B-swizzled layout - no routed buffer.
//   warp 4      TMEM allocator and MMA issuer: one thread issues
//               tcgen05.mma.cta_group::1.kind::f16 (M=128, N<=256, K=16),
//               fp32 accumulators in TMEM, two accumulator buffers so the
//               epilogue of tile i overlaps the main loop of tile i+1 (one
//               buffer of 512 columns in the wide tiles below).
//   warps 5-8   epilogue (5-12 in the wide up, down and dX tiles, four per
//               128-row half): tcgen05.ld of the accumulator rows and the
//               fused per-row work (SwiGLU, gate-weighted combine, SwiGLU
//               backward with the gate gradients, plain stores).
// The CTAs claim tiles from a per-launch counter (weight-gradient tiles in
// descending order of expert load), so skewed expert loads balance.
//
// Wide tiles (up, down with stored H and dX from 32 k-blocks a tile; weight
// gradients from 4,096 routed rows per expert): one CTA takes 256
// output rows, as two M=128 MMAs per 16-deep step that share every B tile,
// into one 512-column accumulator.  A k-block then brings 64 KB for
// 8.4 MFLOP instead of 48 KB for 4.2; the price is that the epilogue is not
// overlapped with the next tile's main loop (there is no second
// accumulator), which the dH stage, with its heavy epilogue, does not repay.
//
// Paired stages (dH, when the reduction is at least 64 k-blocks long): the
// kernel runs as clusters of two CTAs that take two 128-row tiles of one
// expert at the same n-tile.  Both need the same weight tiles: each CTA
// loads half of the boxes and multicasts them to both, halving the weight
// bytes each SM pulls from L2.  A stage is free again once both CTAs' MMAs
// have consumed it (their commits arrive in both CTAs), and the leader
// (rank 0) claims the pair tiles and posts them into both CTAs' tile queues.
//
// Row space: an expert's routed rows form a segment of a padded row space,
// [pad_off[e], pad_off[e+1]), 256-row aligned, so every 128-row M tile (and
// every aligned pair of them: a wide tile, or a cluster pair's tiles)
// belongs to one expert.  Row q of expert e with i = q - pad_off[e] < n_e is
// routed row off[e]+i of token expert_token_indices[off[e]+i]; padding rows
// gather a valid token and are zero where they feed a reduction.
//
// Stage                          A (M x K)                B (K x N)             epilogue
//  UP_SWIGLU  a,b = X W1,X W2    x rows via D1 (gather)   [W1_e | W2_e] tiles   A, B (saved)
//  UP_SILU    a = X W1           x rows via D1            W1_e                  A (saved)
//  DOWN_H     Y = H W3           H rows                   W3_e                  y32[t] += g Y   (red.add)
//  DOWN_*     Y = H W3           H = SiLU(A)*B, from      W3_e                  y32[t] += g Y   (red.add)
//                                the saved A, B tiles
//  DH_*       dH = dY W3^T       dY rows via D1           W3_e (K-major)        dA, dB (SwiGLU bwd), Hg or row gates
//  DX         [dA|dB][W1|W2]^T   dAB rows                 W1_e^T then W2_e^T    dX32[t] += .    (red.add)
//  DW12/DW1   X^T [dA|dB]        x rows via D1 along K    dAB rows (MN-major)   dW1, dW2
//  DW3_H      Hg^T dY            Hg rows (MN-major)       dY rows via D1        dW3
//  DW3_*      Hg^T dY            Hg = g*SiLU(A)*B, from   dY rows via D1        dW3
//                                the saved A, B (MN-major)
//
// By default the up-projection epilogue stores H = SiLU(a) b and the dH
// epilogue Hg = g SiLU(A) B for the down projection and dW3.  With
// MOEBLAZE_RECOMPUTE_H neither is ever written to global memory: DOWN_* and
// DW3_* load the saved A (and B) tiles by TMA and eight transform warps
// recompute the A operand in shared memory, in place, before the tensor
// cores read it (SiLU(a) = a/2 (1 + tanh(a/2)) with tanh.approx).  Each
// stage of the SwiGLU variants also holds the saved-B tile, so their ring
// has 3 stages of 64 KB.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// kErrTimeout in the device error word, drains its own copies and MMAs with
// bounded waits, frees TMEM and returns.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace moeblaze {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_MAX_BYTES = 256 * BK * 2;     // 32 KB
constexpr int PRODUCER_WARPS = 4;
constexpr int PRODUCER_THREADS = PRODUCER_WARPS * 32;
constexpr int TMEM_COLS = 512;                // two 128 x 256 fp32 accumulators
// epilogue staging for TMA stores: a 32 KB area of buffers of 32 rows x 32
// bf16 (64-byte swizzle), a ring of them per epilogue warp
constexpr int EPI_BUF_BYTES = 32 * 64;
constexpr int EPI_STAGE_BYTES = 16 * EPI_BUF_BYTES;  // 32 KB
// Launch variants of a stage: one CTA a tile, clusters of two CTAs sharing
// the weight tiles (row stages), or wide tiles.
enum Variant : int { SINGLE = 0, PAIRED = 1, WIDE = 2 };
constexpr int BAR_BYTES = 512;                // mbarriers, TMEM address, abort flag, tile queue
// Tiles are claimed dynamically: each CTA takes its first two tiles by its
// index and every further one from a global counter, two tiles ahead of
// use, and passes the ids to its MMA and epilogue warps through a queue of
// TQ slots in shared memory.
constexpr int TQ = 8;

// DOWN_H / DW3_H read the H / Hg the up-projection / dH epilogue stored;
// DOWN_SWIGLU, DOWN_SILU, DW3_SWIGLU, DW3_SILU recompute them from the saved
// A (and B) tiles (MOEBLAZE_RECOMPUTE_H).
enum Mode : int {
  UP_SWIGLU = 0, UP_SILU, DOWN_H, DOWN_SWIGLU, DOWN_SILU, DH_SWIGLU, DH_SILU, DX, DW12, DW1, DW3_H, DW3_SWIGLU, DW3_SILU
};

__host__ __device__ constexpr bool is_down(int m) { return m == DOWN_H || m == DOWN_SWIGLU || m == DOWN_SILU; }
__host__ __device__ constexpr bool is_dw3(int m) { return m == DW3_H || m == DW3_SWIGLU || m == DW3_SILU; }
// stages whose A operand is recomputed from the saved A (and B) tiles
__host__ __device__ constexpr bool is_fused(int m) {
  return m == DOWN_SWIGLU || m == DOWN_SILU || m == DW3_SWIGLU || m == DW3_SILU;
}
__host__ __device__ constexpr bool fused_sw(int m) { return m == DOWN_SWIGLU || m == DW3_SWIGLU; }
__host__ __device__ constexpr bool is_wgrad(int m) { return m == DW12 || m == DW1 || is_dw3(m); }
// stages that can run as clusters of two CTAs sharing (multicasting) the
// weight tiles; the host pairs them when the reduction is long
__host__ __device__ constexpr bool pairable(int m) { return m == DH_SWIGLU || m == DH_SILU; }
// Pairing pays off on long reductions with many tiles (measured: the
// Mixtral-like layer's dH 6% faster); on a small layer the pairs' lockstep
// costs more than the shared loads save.  The up projection, the stored-H
// down projection and dX take wide tiles instead (faster there than pairs:
// down 46.9 -> 33.8 ms, dX 84.1 -> 66.8 ms on the Mixtral-like layer).
constexpr int kPairMinKblocks = 64;
constexpr int kPairMinTilesPerSm = 16;
inline bool pair_stage(int kblocks, int64_t tiles) {
  return kblocks >= kPairMinKblocks && tiles >= (int64_t)kPairMinTilesPerSm * sm_count();
}
// Wide tiles for the row stages from 32 k-blocks a tile and 4 (128-row)
// tiles per SM (measured against pair_stage's 64 and 16: the SiLU layer's
// down 0.251 -> 0.223 ms and dX 0.243 -> 0.225 ms, the 64-expert layer's up
// 3.93 -> 3.72 ms and dX 3.60 -> 3.40 ms).
constexpr int kWideMinKblocks = 32;
constexpr int kWideMinTilesPerSm = 4;
inline bool wide_rows(int kblocks, int64_t tiles) {
  return kblocks >= kWideMinKblocks && tiles >= (int64_t)kWideMinTilesPerSm * sm_count();
}
// Warp roles: producers 0-3, in the fused stages eight transform warps
// 4-11, then the MMA warp and four epilogue warps.
__host__ __device__ constexpr int helper_warps(int m) { return is_fused(m) ? 8 : 0; }
__host__ __device__ constexpr int mma_warp(int m) { return PRODUCER_WARPS + helper_warps(m); }
// Epilogue warps: eight in the wide row stages with a stored or combined
// output (one set of four per 128-row half of the tile, so the epilogue
// their single accumulator leaves exposed takes half as long), else four.
// Their TMA-store staging area stays 32 KB: two buffers a warp instead of
// four.
__host__ __device__ constexpr int epi_warps(int m, int v) {
  return v == WIDE && (m == UP_SWIGLU || m == UP_SILU || m == DOWN_H || m == DX) ? 8 : 4;
}
__host__ __device__ constexpr int num_threads(int m, int v = SINGLE) { return (mma_warp(m) + 1 + epi_warps(m, v)) * 32; }
// threads that recompute the A operand of a fused stage
__host__ __device__ constexpr int transform_threads(int m) { return helper_warps(m) * 32; }
// Wide weight-gradient tiles: 256 output rows a CTA, as two M=128 MMAs that
// share every B tile, into one 512-column accumulator (no second buffer: the
// epilogue runs once per reduction, which is long when this is chosen).  A
// k-block then brings 64 KB for 8.4 MFLOP instead of 48 KB for 4.2.
__host__ __device__ constexpr bool widenable(int m) {
  return m == DW12 || m == DW1 || m == DW3_H || m == UP_SWIGLU || m == UP_SILU || m == DOWN_H || m == DX;
}
// Measured: from 4,096 routed rows per expert (64 k-blocks a tile) the wide
// tiles are 20-23% faster on dW1 (dW1 || dW2) and dW3 than 128-row tiles.
constexpr int64_t kWideMinRows = 4096;  // routed rows per expert (on average) from which wide tiles are used
// out_rows: rows of the weight gradient.  A last tile of 128 rows is allowed
// where the A operand comes by TMA (dW3: the rows past the end load as zeros
// and are not stored); the gathered A of dW1 needs whole 256-row tiles.
inline bool wide_stage(const moeblaze_shape& s, int out_rows, bool half_tail_ok) {
  return out_rows % (half_tail_ok ? BM : 2 * BM) == 0 && (int64_t)s.L * s.K >= kWideMinRows * s.E;
}
// The ring: 4 stages of A (16 KB) + B operand (32 KB); the fused SwiGLU
// stages add the saved-B tile (16 KB) to every stage and keep 3 of them;
// wide tiles keep 3 stages of A (32 KB) + B (32 KB).  The fused stages and
// the weight-gradient stages need no epilogue staging area.
__host__ __device__ constexpr int a_bytes_of(int v) { return v == WIDE ? 2 * A_BYTES : A_BYTES; }
__host__ __device__ constexpr int stages_of(int m, int v = SINGLE) { return fused_sw(m) || v == WIDE ? 3 : STAGES; }
__host__ __device__ constexpr int stage_bytes_of(int m, int v = SINGLE) {
  return a_bytes_of(v) + B_MAX_BYTES + (fused_sw(m) ? A_BYTES : 0);
}
__host__ __device__ constexpr int epi_bytes_of(int m, int v = SINGLE) {
  return is_fused(m) || (v == WIDE && is_wgrad(m)) ? 0 : EPI_STAGE_BYTES;
}
__host__ __device__ constexpr int smem_bytes_of(int m, int v = SINGLE) {
  return stages_of(m, v) * stage_bytes_of(m, v) + epi_bytes_of(m, v) + 1024 + BAR_BYTES;
}
static_assert(smem_bytes_of(DW12, WIDE) <= 232448 && smem_bytes_of(UP_SWIGLU, WIDE) <= 232448,
              "wide ring exceeds shared memory");
__host__ __device__ constexpr bool is_dual(int m) { return m == UP_SWIGLU || m == DW12; }
__host__ __device__ constexpr bool a_mn_major(int m) { return is_wgrad(m); }
__host__ __device__ constexpr bool b_k_major(int m) { return m == DH_SWIGLU || m == DH_SILU || m == DX; }
// columns per n-tile (per branch for the dual stages)
__host__ __device__ constexpr int tile_n(int m) { return is_dual(m) ? 128 : 256; }

struct Params {
  CUtensorMap tmA;
  CUtensorMap tmB0;
  CUtensorMap tmB1;
  CUtensorMap tmO0;  // bf16 outputs written by TMA stores (up: A, B, H; dH: dA|dB, Hg)
  CUtensorMap tmO1;
  CUtensorMap tmO2;
  CUtensorMap tmX;   // fused SwiGLU stages: the saved B, same boxes as tmA
  const int32_t* D1;
  const int32_t* D2;
  const int32_t* D3;
  const float* gates;
  MetaView meta;
  int64_t L;
  int d, h, E, K;
  int N;            // output columns (per branch for dual stages)
  int kblocks;      // row stages: reduction length / 64
  int ksplit;       // DX: k-blocks taken from W1 before switching to W2
  int n_tiles;
  int m_tiles_w;    // weight-gradient stages: output rows / 128
  int64_t total_w;  // weight-gradient stages: number of tiles
  __nv_bfloat16* o0;
  __nv_bfloat16* o1;
  __nv_bfloat16* o2;
  const __nv_bfloat16* i0;
  const __nv_bfloat16* i1;
  float* acc32;
  const __nv_bfloat16* gsrc;  // gathered tensor (x or dY), rows of gld elements
  int gld;
  float* dg;                   // dH stage: gate gradients (L,K) fp32, or null
  float* rowg;                 // gate of every padded row (0 for padding rows), recompute mode: written by
                               // the down projection, read by the backward's DW3
  uint64_t wait_ns;            // limit of every bounded wait (kTimeoutNs unless a test sets a shorter one)
  int withhold;                // test of the failure path (DOWN_H): the first stage of each CTA's first
                               // tile is never issued, so the MMA's wait for it runs out
  unsigned long long* sched;  // tile counter of this launch (zero at launch)
};

// Writes this warp's 32 rows x 32 columns (lane = row, v = its 32 values;
// zeros where !valid) to element (col, row0) of `map` through the warp's
// staging ring: the lanes fill a 64-byte-swizzled 2 KB buffer, fence it for
// the async proxy, and lane 0 issues one TMA store (one bulk group each).
struct StoreRing {
  uint32_t base;
  int slot;
};
template <int RING>
__device__ __forceinline__ void staged_store(StoreRing& ring, const CUtensorMap* map, int col, int row0, const float* v,
                                             bool valid, int lane) {
  const uint32_t buf = ring.base + ring.slot * EPI_BUF_BYTES;
  if (lane == 0) bulk_wait_read<RING - 1>();  // this buffer's previous store has been read
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
      u.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
      u.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
      u.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
      u.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
    }
    st_shared_v4(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4), u);
  }
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, col, row0);
    bulk_commit();
  }
  ring.slot = (ring.slot + 1) % RING;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ float fast_sigmoid(float a) { return __fdividef(1.0f, 1.0f + __expf(-a)); }

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
// g * SiLU(a) * b on two bf16 pairs (a, b packed bf16x2), fp32 arithmetic,
// SiLU(a) = h (1 + tanh h) with h = a/2; the result rounded to bf16x2.
template <bool GATED_B, bool GATED_ROW>
__device__ __forceinline__ uint32_t silu_mul2(uint32_t a, uint32_t b, float2 g) {
  const float2 av = make_float2(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u));
  const float2 h = __fmul2_rn(av, make_float2(0.5f, 0.5f));
  const float2 t = make_float2(tanh_approx(h.x), tanh_approx(h.y));
  float2 r = __ffma2_rn(h, t, h);  // SiLU(a)
  if constexpr (GATED_B) r = __fmul2_rn(r, make_float2(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u)));
  if constexpr (GATED_ROW) r = __fmul2_rn(r, g);
  return pack_bf16x2(r.x, r.y);
}
// One transform thread's share (tt = 0..255: the producer warps, then the
// helper warps) of a fused stage's A-operand tile, in place: chunks
// tt + 256 i (i = 0..3) of the tile's 1024 16-byte chunks.  sA holds the
// saved A tile, sX the saved B tile at the same positions (SwiGLU).  For DW3
// the tile is MN-major (two boxes of 64 k-block rows x 128 bytes), so chunk
// tt + 256 i lies in row tt/8 + 32 (i % 2) of the k-block, whose gate is
// g2[i % 2]; the down projection applies its gate in the epilogue.
template <int MODE>
__device__ __forceinline__ void transform_tile(uint32_t sA, uint32_t sX, int tt, const float* g2) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t off = (uint32_t)(tt + 256 * i) * 16u;
    const uint4 a = ld_shared_v4(sA + off);
    uint4 b = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (fused_sw(MODE)) b = ld_shared_v4(sX + off);
    const float gs = is_dw3(MODE) ? g2[i & 1] : 1.f;
    const float2 g = make_float2(gs, gs);
    uint4 o;
    o.x = silu_mul2<fused_sw(MODE), is_dw3(MODE)>(a.x, b.x, g);
    o.y = silu_mul2<fused_sw(MODE), is_dw3(MODE)>(a.y, b.y, g);
    o.z = silu_mul2<fused_sw(MODE), is_dw3(MODE)>(a.z, b.z, g);
    o.w = silu_mul2<fused_sw(MODE), is_dw3(MODE)>(a.w, b.w, g);
    st_shared_v4(sA + off, o);
  }
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// store 32 consecutive fp32 values as bf16 (64 bytes, 16-byte aligned)
__device__ __forceinline__ void store_row32(__nv_bfloat16* p, const float* v) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    q[i] = u;
  }
}
__device__ __forceinline__ void store_zero32(__nv_bfloat16* p) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void unpack_row32(const uint4* q, float* v) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = q[i];
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    v[8 * i + 0] = a.x; v[8 * i + 1] = a.y; v[8 * i + 2] = b.x; v[8 * i + 3] = b.y;
    v[8 * i + 4] = c.x; v[8 * i + 5] = c.y; v[8 * i + 6] = d.x; v[8 * i + 7] = d.y;
  }
}
__device__ __forceinline__ void load_row32(const __nv_bfloat16* p, float* v) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u = q[i];
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    v[8 * i + 0] = a.x; v[8 * i + 1] = a.y; v[8 * i + 2] = b.x; v[8 * i + 3] = b.y;
    v[8 * i + 4] = c.x; v[8 * i + 5] = c.y; v[8 * i + 6] = d.x; v[8 * i + 7] = d.y;
  }
}

// ------------------------------------------------------------------ tile decode
struct Tile {
  int e;        // expert
  int row0;     // row stages: first padded row; weight stages: first output row (m0)
  int n0;       // first output column (per branch)
  int nw;       // columns in this tile (per branch)
  int kblocks;  // k-blocks of 64
  int pad0;     // pad_off[e]
  int off;      // expert_token_offsets[e]
  int n_e;      // tokens routed to e
};

// Tile `tile` of the launch.  In the paired stages a tile id names a pair of
// 128-row tiles of one expert (a 256-row slice of its padded segment) at one
// n-tile, and `rank` picks this CTA's half.
template <int MODE, bool PAIR, bool WIDE_T = false>
__device__ __forceinline__ Tile decode(const Params& p, int64_t tile, int num_mt, int rank) {
  Tile t;
  constexpr int TN = tile_n(MODE);
  constexpr int PM = PAIR || WIDE_T ? 2 : 1;
  int nt;
  if constexpr (is_wgrad(MODE)) {
    const int64_t per_e = (int64_t)p.m_tiles_w * p.n_tiles;
    const int rank = (int)(tile / per_e);
    const int r = (int)(tile % per_e);
    // groups of GW m-tiles walk the n-tiles together: the CTAs running at
    // once then share fewer, more reused A and B slices in L2.  Measured on
    // the Mixtral-like layer's dW1 || dW2 with 256-row tiles: DRAM reads of
    // 544 GB a launch with groups of 16 (all of d), 173 GB with 8, 242 GB
    // with 4 (97.6, 78.7 and 81.3 ms); 128-row tiles keep 16.
    constexpr int GW = WIDE_T ? 8 : 16;
    const int g = r / (GW * p.n_tiles);
    const int gw = min(GW, p.m_tiles_w - g * GW);
    const int rr = r - g * GW * p.n_tiles;
    const int mt = g * GW + rr % gw;
    nt = rr / gw;
    t.e = p.meta.order[rank];
    t.row0 = mt * BM * (WIDE_T ? 2 : 1);
    t.pad0 = p.meta.pad_off[t.e];
    t.kblocks = (p.meta.pad_off[t.e + 1] - t.pad0) / BK;
  } else {
    // groups of 16 m-tiles (8 pairs) walk the n-tiles together, so the weight
    // tiles they share stay in L2
    constexpr int GM = 16 / PM;
    const int nmu = num_mt / PM;
    const int64_t per_g = (int64_t)GM * p.n_tiles;
    const int g = (int)(tile / per_g);
    const int r = (int)(tile % per_g);
    const int gm = min(GM, nmu - g * GM);
    const int mt = (g * GM + r % gm) * PM + (PM == 2 ? rank : 0);
    nt = r / gm;
    t.e = p.meta.tile_expert[mt];
    t.row0 = mt * BM;
    t.pad0 = p.meta.pad_off[t.e];
    t.kblocks = p.kblocks;
  }
  t.off = p.D2[t.e];
  t.n_e = p.D2[t.e + 1] - t.off;
  t.n0 = nt * TN;
  t.nw = min(TN, p.N - t.n0);
  return t;
}

// token of padded row q of the tile's expert (clamped to the last routed row)
__device__ __forceinline__ int row_token(const Params& p, const Tile& t, int q) {
  if (t.n_e == 0) return 0;  // an expert with no tokens: nothing is read for it
  int i = q - t.pad0;
  if (i >= t.n_e) i = t.n_e - 1;
  if (i < 0) i = 0;
  return p.D1[t.off + i];
}

// gate of (token, expert) and its slot k (token_expert_indices[tok, k] == e)
__device__ __forceinline__ float gate_of(const Params& p, int tok, int e, int* slot = nullptr) {
  const int64_t b = (int64_t)tok * p.K;
  for (int k = 0; k < p.K; ++k)
    if (p.D3[b + k] == e) {
      if (slot) *slot = k;
      return p.gates[b + k];
    }
  if (slot) *slot = 0;
  return 0.f;
}

// ------------------------------------------------------------------ kernel
// Operands fetched by the cp.async gather producer (rows picked through
// expert_token_indices); every other operand tile comes by tiled TMA.
__host__ __device__ constexpr bool cp_a(int m) {
  return m == UP_SWIGLU || m == UP_SILU || m == DH_SWIGLU || m == DH_SILU || m == DW12 || m == DW1;
}
__host__ __device__ constexpr bool cp_b(int m) { return is_dw3(m); }

template <int MODE, int VAR>
__global__ void __launch_bounds__(num_threads(MODE, VAR), 1) moe_gemm_kernel(const __grid_constant__ Params p) {
  constexpr bool PAIR = VAR == PAIRED;
  // WIDE: 256-row weight-gradient tiles (two M=128 MMAs a k-step, one accumulator)
  constexpr bool WIDE_T = VAR == WIDE;
  static_assert(!WIDE_T || widenable(MODE), "stage has no wide tiles");
  constexpr int NACC = WIDE_T ? 1 : 2;  // accumulator buffers in TMEM
  constexpr int AB = a_bytes_of(VAR);   // A part of a stage
  constexpr int EW = epi_warps(MODE, VAR);                 // epilogue warps
  constexpr int ER = EPI_STAGE_BYTES / (EW * EPI_BUF_BYTES);  // staging buffers per epilogue warp
  constexpr bool CPA = cp_a(MODE), CPB = cp_b(MODE), CP = CPA || CPB;
  // FUSED: transform warps recompute the A operand from the saved tiles
  constexpr bool FUSED = is_fused(MODE);
  constexpr int MMA_WARP = mma_warp(MODE);
  constexpr int NST = stages_of(MODE, VAR), SB = stage_bytes_of(MODE, VAR);
  constexpr int LAG = NST - 2;  // cp.async groups a producer thread keeps in flight
  // PAIR: clusters of two CTAs share the weight tiles (multicast) and the
  // tile queue (filled by rank 0)
  static_assert(!PAIR || pairable(MODE), "stage cannot run paired");
  const int rank = PAIR ? (int)cluster_rank() : 0;
  const int64_t cta0 = PAIR ? blockIdx.x / 2 : blockIdx.x;      // cluster (pair) index
  const int64_t ncta = PAIR ? gridDim.x / 2 : gridDim.x;        // clusters (pairs) in the grid
  // A dispatch built for another (L, E, K) lays out its tables differently:
  // record the mismatch and read none of them (every thread reads the same
  // three header words, so the whole CTA leaves here together, before any
  // barrier or TMEM allocation).
  if (!meta_matches(p.meta.hdr, p.L, p.E, p.K)) {
    if (threadIdx.x == 0) atomicOr(p.meta.err, kErrShapeMismatch);
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NST * SB + epi_bytes_of(MODE, VAR));
  // bars: full[0..3], empty[4..7], tmem_full[8..9], tmem_empty[10..11], drain[12],
  // loaded[48..51] (fused stages: the TMA part of a stage has landed)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_s = reinterpret_cast<volatile int*>(bars + 17);
  // tile-id queue: ids at bars[24 + i], full barriers bars[32 + i], empty barriers bars[40 + i]
  volatile long long* tq = reinterpret_cast<volatile long long*>(bars + 24);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      // full: the gathering producer threads (cp.async stages), the transform
      // warps (fused stages), else thread 0's arrive.expect_tx
      mbar_init(bar(s), FUSED || CP ? (CP ? PRODUCER_THREADS : 0) + transform_threads(MODE) : 1);
      // empty: this CTA's MMA commit (and the peer's, when the pair shares the stage's weight tiles)
      mbar_init(bar(4 + s), PAIR ? 2 : 1);
      mbar_init(bar(48 + s), 1);
    }
    mbar_init(bar(8), 1);
    mbar_init(bar(9), 1);
    mbar_init(bar(10), 32 * EW);
    mbar_init(bar(11), 32 * EW);
    mbar_init(bar(12), 1);
    for (int i = 0; i < TQ; ++i) {
      mbar_init(bar(32 + i), 1);
      // readers of a queue slot: the producer warps (thread 0 alone in the
      // TMA-only stages), the transform warps (fused stages), the MMA thread
      // and the four epilogue warps; in a pair rank 0's slot is also freed by
      // the peer's readers (rank 1 posts nothing)
      mbar_init(bar(40 + i), ((CP ? PRODUCER_WARPS : 1) + helper_warps(MODE) + 1 + EW) * (PAIR ? 2 : 1));
    }
    *abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the peer's barriers exist before any multicast or remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_mt = is_wgrad(MODE) ? 0 : *p.meta.num_m_tiles;
  const int64_t total = is_wgrad(MODE) ? p.total_w : (int64_t)(num_mt / (PAIR || WIDE_T ? 2 : 1)) * p.n_tiles;
  int32_t* err = p.meta.err;
  const uint64_t lim = p.wait_ns;

  // queue position j lives in slot j % TQ, phase (j / TQ) & 1
  auto q_post = [&](int j, long long id) -> bool {  // thread 0 (of rank 0 in a pair)
    const int sl = j % TQ;
    if (!wait_bounded<PAIR>(bar(40 + sl), (uint32_t)((j / TQ) & 1) ^ 1u, abort_s, err, lim)) return false;
    tq[sl] = id;
    mbar_arrive(bar(32 + sl));
    if constexpr (PAIR) {
      // the same id in the peer's slot, then its full barrier (release at cluster scope)
      st_cluster_u64(peer_addr(smem_u32((const void*)(tq + sl)), 1u), (unsigned long long)id);
      mbar_arrive_cluster(peer_addr(bar(32 + sl), 1u));
    }
    return true;
  };
  auto q_take = [&](int j) -> long long {  // one thread per reader; -1 once the CTA gives up
    const int sl = j % TQ;
    if (!wait_bounded<PAIR>(bar(32 + sl), (uint32_t)(j / TQ) & 1u, abort_s, err, lim)) return -1;
    const long long id = tq[sl];
    if (PAIR && rank == 1) mbar_arrive_cluster(peer_addr(bar(40 + sl), 0u));  // rank 0 owns the slots
    else mbar_arrive(bar(40 + sl));
    return id;
  };
  // tile of queue position j >= 2 (positions 0 and 1 are this CTA's (pair's)
  // first two: cta0 and cta0 + ncta)
  auto claim = [&]() -> long long { return 2ll * ncta + (long long)atomicAdd(p.sched, 1ull); };

  if (warp < PRODUCER_WARPS) {
    // ================================================================ producer
    // Thread 0 issues the tiled TMA loads.  In the gather stages all 128
    // producer threads also copy the gathered operand with 16-byte cp.async
    // straight into the 128B-swizzled layout (8 consecutive threads cover one
    // 128-byte row segment), keep LAG groups in flight, and arrive on the
    // stage's full barrier once their copies of it have landed and been
    // fenced for the tensor cores (async proxy).  In the fused stages the
    // saved A (and B) tiles go to the stage's `loaded` barrier instead, for
    // the transform warps, which then complete the full barrier.
    const int pt = threadIdx.x;
    if (CP || pt == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t armed = 0, armed_par = 0;
      int inflight = 0;
      bool ok = true;
      const int c8 = pt & 7;   // 16-byte chunk of a 128-byte row this thread copies
      const int r16 = pt >> 3; // row offset 0..15 within a group of 16 rows
      // The routed-row tokens of the next tile are loaded while this tile's
      // k-blocks are issued, so a tile change costs no load latency.
      constexpr int NR = AB / 2048;  // gathered rows per thread (row stages): 8, wide tiles 16
      int rtok[NR], wtok[4], rnext[NR], wfirst[4];
      auto load_tile_tokens = [&](const Tile& tt, int* rr, int* ww) {
        if constexpr (CP && !is_wgrad(MODE)) {
#pragma unroll
          for (int it = 0; it < NR; ++it) rr[it] = row_token(p, tt, tt.row0 + it * 16 + r16);
        }
        if constexpr (CP && is_wgrad(MODE)) {
#pragma unroll
          for (int i = 0; i < 4; ++i) ww[i] = row_token(p, tt, tt.pad0 + i * 16 + r16);
        }
      };
      // the producer warps read queue position j + 1 while they issue tile j
      auto take = [&](int j) -> long long {
        long long id = 0;
        if constexpr (CP) {
          if (lane == 0) id = q_take(j);
          id = __shfl_sync(0xffffffffu, id, 0);
        } else {
          id = q_take(j);
        }
        return id;
      };
      if (pt == 0 && rank == 0 && q_post(0, cta0)) q_post(1, (long long)cta0 + ncta);
      long long tile = take(0);
      Tile t;
      if (tile >= 0 && tile < total) {
        t = decode<MODE, PAIR, WIDE_T>(p, tile, num_mt, rank);
        load_tile_tokens(t, rtok, wtok);
      }
      ok = tile >= 0;
      for (int j = 0; ok && tile < total; ++j) {
        long long pending = 0;
        if (pt == 0 && rank == 0) pending = claim();  // for position j + 2, posted after this tile's loads are issued
        const long long ntile = take(j + 1);
        if (ntile < 0) {
          ok = false;
          break;
        }
        Tile tn;
        if (ntile < total) {
          tn = decode<MODE, PAIR, WIDE_T>(p, ntile, num_mt, rank);
          load_tile_tokens(tn, rnext, wfirst);
        }
        const int nmma = is_dual(MODE) ? 2 * t.nw : t.nw;
        if constexpr (CP) {
          // A tile without k-blocks (an expert with no tokens) issues no
          // stage that would release the arrivals still held back, and the
          // queue may make this warp wait on the epilogue, which needs them:
          // deliver them now.
          if (t.kblocks == 0 && inflight > 0) {
            cp_async_wait<0>();
            fence_proxy_async();
            for (int i = inflight; i > 0; --i) mbar_arrive(bar((s + NST - i) % NST));
            inflight = 0;
          }
        }
        for (int kb = 0; kb < t.kblocks; ++kb) {
          if constexpr (CP) {
            // every lane of the four producer warps is here: lane 0 waits, the warp follows
            if (lane == 0) ok = wait_bounded(bar(4 + s), ph ^ 1u, abort_s, err, lim);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          } else {
            // thread 0 runs this loop alone: no warp-collective operations here
            ok = wait_bounded(bar(4 + s), ph ^ 1u, abort_s, err, lim);
          }
          if (!ok) break;
          const uint32_t full = bar(s);
          const uint32_t loaded = bar(48 + s);
          const uint32_t sA = smem_base + s * SB;
          const uint32_t sB = sA + AB;
          const uint32_t sX = sB + B_MAX_BYTES;  // fused SwiGLU: the saved-B tile
          const int k0 = kb * BK;
          int wnext[4];
          if constexpr (CP && is_wgrad(MODE)) {
            if (kb + 1 < t.kblocks) {
#pragma unroll
              for (int i = 0; i < 4; ++i) wnext[i] = row_token(p, t, t.pad0 + k0 + BK + i * 16 + r16);
            }
          }
          // test of the failure path: the down projection leaves the first
          // stage of this CTA's first tile empty; nothing ever completes its
          // full barrier
          const bool withheld = MODE == DOWN_H && p.withhold && j == 0 && kb == 0;
          if (pt == 0 && !withheld) {
            // ---------------- tiled TMA part of the stage
            if constexpr (FUSED) {
              const uint32_t tma_bytes = (uint32_t)A_BYTES + (fused_sw(MODE) ? (uint32_t)A_BYTES : 0u) +
                                         (is_down(MODE) ? (uint32_t)(nmma * BK * 2) : 0u);
              mbar_expect_tx(loaded, tma_bytes);
            } else {
              const uint32_t tma_bytes = (CPA ? 0u : (uint32_t)AB) + (CPB ? 0u : (uint32_t)(nmma * BK * 2));
              if (CP) mbar_expect_tx_only(full, tma_bytes);
              else mbar_expect_tx(full, tma_bytes);
            }
            armed |= 1u << s;
            armed_par = (armed_par & ~(1u << s)) | (ph << s);
            // box j of the weight tile both CTAs of a pair share: the CTA of
            // rank j % 2 loads it for both (multicast); unpaired, this CTA
            auto wbox = [&](int jb, uint32_t dst, const CUtensorMap* m, int c0, int c1, uint32_t b) {
              if constexpr (PAIR) {
                if ((jb & 1) == rank) tma_load_2d_mc(dst, m, c0, c1, b, (uint16_t)0x3);
              } else {
                tma_load_2d(dst, m, c0, c1, b);
              }
            };
            if constexpr (MODE == DOWN_H) {
#pragma unroll
              for (int a = 0; a < AB / A_BYTES; ++a) tma_load_2d(sA + a * A_BYTES, &p.tmA, k0, t.row0 + a * BM, full);
            } else if constexpr (MODE == DX) {
              // [dA | dB] along K: the first ksplit k-blocks from dA, the rest from dB
              const bool second = kb >= p.ksplit;
#pragma unroll
              for (int a = 0; a < AB / A_BYTES; ++a)
                tma_load_2d(sA + a * A_BYTES, second ? &p.tmX : &p.tmA, second ? k0 - p.ksplit * BK : k0,
                            t.row0 + a * BM, full);
            } else if constexpr (MODE == DW3_H) {
#pragma unroll
              for (int a = 0; a < AB / 8192; ++a) tma_load_2d(sA + 8192 * a, &p.tmA, t.row0 + 64 * a, t.pad0 + k0, full);
            } else if constexpr (is_down(MODE)) {
              tma_load_2d(sA, &p.tmA, k0, t.row0, loaded);
              if constexpr (fused_sw(MODE)) tma_load_2d(sX, &p.tmX, k0, t.row0, loaded);
            } else if constexpr (is_dw3(MODE)) {
              tma_load_2d(sA, &p.tmA, t.row0, t.pad0 + k0, loaded);
              tma_load_2d(sA + 8192, &p.tmA, t.row0 + 64, t.pad0 + k0, loaded);
              if constexpr (fused_sw(MODE)) {
                tma_load_2d(sX, &p.tmX, t.row0, t.pad0 + k0, loaded);
                tma_load_2d(sX + 8192, &p.tmX, t.row0 + 64, t.pad0 + k0, loaded);
              }
            }
            if constexpr (MODE == UP_SWIGLU) {
              wbox(0, sB, &p.tmB0, t.n0, t.e * p.d + k0, full);
              wbox(1, sB + 8192, &p.tmB0, t.n0 + 64, t.e * p.d + k0, full);
              wbox(2, sB + 16384, &p.tmB1, t.n0, t.e * p.d + k0, full);
              wbox(3, sB + 24576, &p.tmB1, t.n0 + 64, t.e * p.d + k0, full);
            } else if constexpr (MODE == UP_SILU) {
              for (int j = 0; j < t.nw / 64; ++j) wbox(j, sB + j * 8192, &p.tmB0, t.n0 + 64 * j, t.e * p.d + k0, full);
            } else if constexpr (is_down(MODE)) {
              const uint32_t wb = FUSED ? loaded : full;
              for (int j = 0; j < t.nw / 64; ++j) wbox(j, sB + j * 8192, &p.tmB0, t.n0 + 64 * j, t.e * p.h + k0, wb);
            } else if constexpr (MODE == DH_SWIGLU || MODE == DH_SILU) {
              for (int j = 0; j < t.nw / 128; ++j)
                wbox(j, sB + j * 16384, &p.tmB0, k0, t.e * p.h + t.n0 + 128 * j, full);
            } else if constexpr (MODE == DX) {
              const bool second = kb >= p.ksplit;
              const CUtensorMap* m = second ? &p.tmB1 : &p.tmB0;
              const int kc = second ? k0 - p.ksplit * BK : k0;
              for (int j = 0; j < t.nw / 128; ++j) wbox(j, sB + j * 16384, m, kc, t.e * p.d + t.n0 + 128 * j, full);
            } else if constexpr (MODE == DW12) {
              tma_load_2d(sB, &p.tmB0, t.n0, t.pad0 + k0, full);
              tma_load_2d(sB + 8192, &p.tmB0, t.n0 + 64, t.pad0 + k0, full);
              tma_load_2d(sB + 16384, &p.tmB1, t.n0, t.pad0 + k0, full);
              tma_load_2d(sB + 24576, &p.tmB1, t.n0 + 64, t.pad0 + k0, full);
            } else if constexpr (MODE == DW1) {
              for (int j = 0; j < t.nw / 64; ++j) tma_load_2d(sB + j * 8192, &p.tmB0, t.n0 + 64 * j, t.pad0 + k0, full);
            }
          }
          if constexpr (CP) {
            // ---------------- gathered part of the stage
            if constexpr (!is_wgrad(MODE)) {
              // K-major A: 128 (wide tiles 256) routed rows x 64 columns of x (or dY)
#pragma unroll
              for (int it = 0; it < NR; ++it) {
                const int r = it * 16 + r16;
                const __nv_bfloat16* src = p.gsrc + (int64_t)rtok[it] * p.gld + k0 + c8 * 8;
                cp_async16(sA + r * 128 + ((c8 ^ (r & 7)) << 4), src);
              }
            } else {
              // MN-major operand gathered along K: 64 routed rows x (atoms of 64 columns)
              const int col0 = CPA ? t.row0 : t.n0;
              const uint32_t dst0 = CPA ? sA : sB;
              const int natoms = CPA ? AB / 8192 : t.nw / 64;
              for (int j = 0; j < natoms; ++j) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int r = i * 16 + r16;
                  const __nv_bfloat16* src = p.gsrc + (int64_t)wtok[i] * p.gld + col0 + 64 * j + c8 * 8;
                  cp_async16(dst0 + j * 8192 + r * 128 + ((c8 ^ (r & 7)) << 4), src);
                }
              }
            }
            cp_async_commit();
            if (inflight == LAG) {
              cp_async_wait<LAG>();
              fence_proxy_async();
              mbar_arrive(bar((s + NST - LAG) % NST));
            } else {
              ++inflight;
            }
          }
          if constexpr (CP && is_wgrad(MODE)) {
            if (kb + 1 < t.kblocks) {
#pragma unroll
              for (int i = 0; i < 4; ++i) wtok[i] = wnext[i];
            }
          }
          if (++s == NST) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        if (pt == 0 && rank == 0) ok = q_post(j + 2, pending);
        if constexpr (CP) {
          if (warp == 0) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        if (!ok) break;
        tile = ntile;
        if (ntile < total) {
          t = tn;
#pragma unroll
          for (int i = 0; i < NR; ++i) rtok[i] = rnext[i];
#pragma unroll
          for (int i = 0; i < 4; ++i) wtok[i] = wfirst[i];
        }
      }
      if constexpr (CP) {
        // the last `inflight` stages: wait for their copies and arrive
        cp_async_wait<0>();
        fence_proxy_async();
        for (int i = inflight; i > 0; --i) mbar_arrive(bar((s + NST - i) % NST));
      }
      if ((!ok || p.withhold) && pt == 0) {
        // give the TMA copies already issued a bounded chance to land
        for (int i = 0; i < NST; ++i)
          if (armed & (1u << i))
            wait_bounded(bar(FUSED ? 48 + i : i), (armed_par >> i) & 1u, nullptr, nullptr, kDrainNs);
      }
    }
  } else if (warp < MMA_WARP) {
    // ================================================================ transform warps
    // Fused stages only: every stage's A operand is recomputed here, in
    // place, from the saved tiles its TMA part brought in.  The warps follow
    // the tile queue and the k-blocks in the producer's order, wait for each
    // stage's `loaded` barrier, recompute their chunks, fence them for the
    // tensor cores and arrive on the full barrier.
    if constexpr (FUSED) {
      const int tt = threadIdx.x - PRODUCER_THREADS;  // 0..255
      int hs = 0;
      uint32_t hph = 0;
      bool ok = true;
      for (int j = 0; ok; ++j) {
        long long tile = 0;
        if (lane == 0) tile = q_take(j);
        tile = __shfl_sync(0xffffffffu, tile, 0);
        if (tile < 0 || tile >= total) break;
        const Tile t = decode<MODE, PAIR, WIDE_T>(p, tile, num_mt, rank);
        for (int kb = 0; kb < t.kblocks; ++kb) {
          float g2[2] = {1.f, 1.f};
          if constexpr (is_dw3(MODE)) {
#pragma unroll
            for (int i = 0; i < 2; ++i) g2[i] = p.rowg[t.pad0 + kb * BK + (tt >> 3) + 32 * i];
          }
          bool got = true;
          if (lane == 0) got = wait_bounded(bar(48 + hs), hph, abort_s, err, lim);
          ok = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
          if (!ok) break;
          // every lane observes the completed phase itself (acquire) before it
          // reads what the TMA wrote; the phase cannot move on before this
          // stage's full barrier, which needs every transform thread
          (void)mbar_try(bar(48 + hs), hph);
          const uint32_t sA = smem_base + hs * SB;
          transform_tile<MODE>(sA, sA + A_BYTES + B_MAX_BYTES, tt, g2);
          fence_proxy_async();
          mbar_arrive(bar(hs));
          if (++hs == NST) { hs = 0; hph ^= 1u; }
        }
      }
    }
  } else if (warp == MMA_WARP) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int abuf = 0;
      uint32_t aph = 0;
      bool ok = true;
      long long tile = q_take(0);
      Tile t;
      if (tile >= 0 && tile < total) t = decode<MODE, PAIR, WIDE_T>(p, tile, num_mt, rank);
      for (int j = 0; ok; ++j) {
        if (tile < 0) {
          ok = false;
          break;
        }
        if (tile >= total) break;
        // The next tile's id and description (dependent loads of the expert
        // tables in the weight stages) are fetched once this tile's first
        // MMAs are issued, so their latency overlaps the tile's main loop.
        long long ntile = -1;
        Tile tn;
        bool fetched = false;
        auto fetch_next = [&]() {
          ntile = q_take(j + 1);
          if (ntile >= 0 && ntile < total) tn = decode<MODE, PAIR, WIDE_T>(p, ntile, num_mt, rank);
          fetched = true;
        };
        const int nmma = is_dual(MODE) ? 2 * t.nw : t.nw;
        const uint32_t idesc = instr_desc(nmma, a_mn_major(MODE), !b_k_major(MODE));
        ok = wait_bounded(bar(10 + abuf), aph ^ 1u, abort_s, err, lim);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dcol = tmem_base + abuf * 256;
        for (int kb = 0; kb < t.kblocks; ++kb) {
          ok = wait_bounded(bar(s), ph, abort_s, err, lim);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sA = smem_base + s * SB;
          const uint32_t sB = sA + AB;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = b_k_major(MODE) ? smem_desc(sB + kk * 32, 16, 1024) : smem_desc(sB + kk * 2048, 8192, 1024);
            if constexpr (WIDE_T) {
              // rows 0-127 and 128-255 of the tile (MN-major A: atoms 0-1 and
              // 2-3; K-major A: 16 KB apart) into accumulator columns 0 and 256
#pragma unroll
              for (int hm = 0; hm < 2; ++hm) {
                const uint64_t ad = a_mn_major(MODE) ? smem_desc(sA + hm * 16384 + kk * 2048, 8192, 1024)
                                                     : smem_desc(sA + hm * 16384 + kk * 32, 16, 1024);
                mma_bf16(dcol + hm * 256, ad, bd, idesc, (kb | kk) ? 1u : 0u);
              }
            } else {
              const uint64_t ad =
                  a_mn_major(MODE) ? smem_desc(sA + kk * 2048, 8192, 1024) : smem_desc(sA + kk * 32, 16, 1024);
              mma_bf16(dcol, ad, bd, idesc, (kb | kk) ? 1u : 0u);
            }
          }
          if constexpr (PAIR) mma_commit_mc(bar(4 + s), (uint16_t)0x3);  // frees the stage in both CTAs
          else mma_commit(bar(4 + s));
          if (++s == NST) { s = 0; ph ^= 1u; }
          if (kb == 0) fetch_next();
        }
        if (!ok) break;
        mma_commit(bar(8 + abuf));
        if (++abuf == NACC) { abuf = 0; aph ^= 1u; }
        if (!fetched) fetch_next();
        tile = ntile;
        t = tn;
      }
      // all MMAs issued by this thread retire before TMEM is released
      mma_commit(bar(12));
      wait_bounded(bar(12), 0, nullptr, nullptr, ok ? lim : kDrainNs);
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter ...
    const int r = quarter * 32 + lane;            // accumulator row of this thread
    const int ew = warp - MMA_WARP - 1;           // epilogue warp 0 .. EW-1
    StoreRing ring{smem_base + NST * SB + ew * ER * EPI_BUF_BYTES, 0};
    int abuf = 0;
    uint32_t aph = 0;
    for (int j = 0;; ++j) {
      long long tile = 0;
      if (lane == 0) tile = q_take(j);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (tile < 0 || tile >= total) break;
      const Tile t = decode<MODE, PAIR, WIDE_T>(p, tile, num_mt, rank);
      // Per-row context that does not depend on the accumulator is fetched
      // before waiting for it, so its latency overlaps the main loop.
      constexpr bool DH = MODE == DH_SWIGLU || MODE == DH_SILU;
      int q = 0, tok = 0, kslot = 0;
      bool valid = false;
      float g = 1.f;
      // wide tiles of the combining stages: the same for row q + 128
      int tok_1 = 0;
      bool valid_1 = false;
      float g_1 = 1.f;
      uint4 nA[4], nB[4];
      if constexpr (!is_wgrad(MODE)) {
        q = t.row0 + r;
        valid = (q - t.pad0) < t.n_e;
        if constexpr (is_down(MODE) || MODE == DX || DH) {
          if (valid) {
            tok = p.D1[t.off + (q - t.pad0)];
            if constexpr (MODE != DX) g = gate_of(p, tok, t.e, &kslot);
          }
        }
        if constexpr (WIDE_T && (is_down(MODE) || MODE == DX)) {
          valid_1 = (q + BM - t.pad0) < t.n_e;
          if (valid_1) {
            tok_1 = p.D1[t.off + (q + BM - t.pad0)];
            if constexpr (MODE != DX) g_1 = gate_of(p, tok_1, t.e);
          }
        }
        if constexpr (DH) {
          if (valid) {
            const uint4* pa = reinterpret_cast<const uint4*>(p.i0 + (int64_t)q * p.h + t.n0);
#pragma unroll
            for (int i = 0; i < 4; ++i) nA[i] = pa[i];
            if constexpr (MODE == DH_SWIGLU) {
              const uint4* pb = reinterpret_cast<const uint4*>(p.i1 + (int64_t)q * p.h + t.n0);
#pragma unroll
              for (int i = 0; i < 4; ++i) nB[i] = pb[i];
              // The rest of this row's A and B pieces (one 128-byte line per
              // 64 columns) are pulled into L2 now, while the accumulator is
              // still being computed; the chunk loads below then hit L2.
              // (Measured: SwiGLU dH 4% faster; no gain with one operand.)
              for (int i = 1; i < t.nw / 64; ++i) {
                prefetch_l2(p.i0 + (int64_t)q * p.h + t.n0 + 64 * i);
                prefetch_l2(p.i1 + (int64_t)q * p.h + t.n0 + 64 * i);
              }
            }
          }
        }
      }
      bool ok = true;
      if (lane == 0) ok = wait_bounded(bar(8 + abuf), aph, abort_s, err, lim);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + abuf * 256;
      const int wrow0 = t.row0 + quarter * 32;    // first row of this warp in the output
      uint32_t ra[32], rb[32];
      float va[32], vb[32];

      if constexpr (!is_wgrad(MODE)) {
        if constexpr (MODE == UP_SWIGLU || MODE == UP_SILU) {
          // wide tiles: rows 128-255 of the tile from accumulator columns
          // 256-511 (with eight epilogue warps, by the second four)
          const int hm0 = EW == 8 ? ew / 4 : 0;
#pragma unroll 1
          for (int hm = hm0; hm < (EW == 8 ? hm0 + 1 : WIDE_T ? 2 : 1); ++hm) {
            const uint32_t tb = tbase + hm * 256;
            const int wr = wrow0 + hm * BM;
            const bool vr = hm == 0 ? valid : (q + BM - t.pad0) < t.n_e;
            if constexpr (MODE == UP_SWIGLU) {
              for (int c = 0; c < t.nw / 32; ++c) {
                MB_TMEM_LD32(tb + 32 * c, ra);
                MB_TMEM_LD32(tb + 128 + 32 * c, rb);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  va[i] = __uint_as_float(ra[i]);
                  vb[i] = __uint_as_float(rb[i]);
                }
                staged_store<ER>(ring, &p.tmO0, t.n0 + 32 * c, wr, va, vr, lane);
                staged_store<ER>(ring, &p.tmO1, t.n0 + 32 * c, wr, vb, vr, lane);
                if (p.o2) {  // H for the down projection (not with MOEBLAZE_RECOMPUTE_H)
                  float vh[32];
#pragma unroll
                  for (int i = 0; i < 32; ++i) vh[i] = va[i] * fast_sigmoid(va[i]) * vb[i];
                  staged_store<ER>(ring, &p.tmO2, t.n0 + 32 * c, wr, vh, vr, lane);
                }
              }
            } else {
              for (int c = 0; c < t.nw / 32; ++c) {
                MB_TMEM_LD32(tb + 32 * c, ra);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) va[i] = __uint_as_float(ra[i]);
                staged_store<ER>(ring, &p.tmO0, t.n0 + 32 * c, wr, va, vr, lane);
                if (p.o2) {  // H = SiLU(a) for the down projection (not with MOEBLAZE_RECOMPUTE_H)
#pragma unroll
                  for (int i = 0; i < 32; ++i) vb[i] = va[i] * fast_sigmoid(va[i]);
                  staged_store<ER>(ring, &p.tmO2, t.n0 + 32 * c, wr, vb, vr, lane);
                }
              }
            }
          }
        } else if constexpr (is_down(MODE) || MODE == DX) {
          // MOEBLAZE_RECOMPUTE_H: the forward keeps every padded row's gate
          // for the backward's dW3 (0 on padding rows); once per row
          if constexpr (is_down(MODE)) {
            if (p.rowg && t.n0 == 0) p.rowg[q] = valid ? g : 0.f;
          }
          // wide tiles: rows 128-255 of the tile from accumulator columns
          // 256-511 (with eight epilogue warps, by the second four)
          const int hm0 = EW == 8 ? ew / 4 : 0;
#pragma unroll 1
          for (int hm = hm0; hm < (EW == 8 ? hm0 + 1 : WIDE_T ? 2 : 1); ++hm) {
            const bool vr = hm == 0 ? valid : valid_1;
            const float gr = hm == 0 ? g : g_1;
            float* dst = p.acc32 + (int64_t)(hm == 0 ? tok : tok_1) * p.d + t.n0;
            for (int c = 0; c < t.nw / 32; ++c) {
              MB_TMEM_LD32(tbase + hm * 256 + 32 * c, ra);
              tmem_wait_ld();
              if (vr) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                  red_add_v4(dst + 32 * c + i, gr * __uint_as_float(ra[i]), gr * __uint_as_float(ra[i + 1]),
                             gr * __uint_as_float(ra[i + 2]), gr * __uint_as_float(ra[i + 3]));
              }
            }
          }
        } else {  // DH_SWIGLU / DH_SILU
          constexpr bool SW = MODE == DH_SWIGLU;
          const int64_t ro = (int64_t)q * p.h + t.n0;              // A, B rows
          const int nch = t.nw / 32;
          float dgp = 0.f;  // this tile's part of <H_row, dY W3^T> = <dY, Y_row>
          for (int c = 0; c < nch; ++c) {
            // chunk c of A (B) was loaded one step ahead; start loading chunk c+1
            uint4 cA[4], cB[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              cA[i] = nA[i];
              if constexpr (SW) cB[i] = nB[i];
            }
            if (valid && c + 1 < nch) {
              const uint4* pa = reinterpret_cast<const uint4*>(p.i0 + ro + 32 * (c + 1));
#pragma unroll
              for (int i = 0; i < 4; ++i) nA[i] = pa[i];
              if constexpr (SW) {
                const uint4* pb = reinterpret_cast<const uint4*>(p.i1 + ro + 32 * (c + 1));
#pragma unroll
                for (int i = 0; i < 4; ++i) nB[i] = pb[i];
              }
            }
            MB_TMEM_LD32(tbase + 32 * c, ra);
            tmem_wait_ld();
            float A[32], B[32], dA[32], dB[32], Hg[32];
            unpack_row32(cA, A);
            if constexpr (SW) unpack_row32(cB, B);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float dH = g * __uint_as_float(ra[i]);
              const float a = A[i];
              const float sg = fast_sigmoid(a);
              const float sl = a * sg;
              const float ds = sg * (1.f + a * (1.f - sg));
              if constexpr (SW) {
                dA[i] = dH * B[i] * ds;
                dB[i] = dH * sl;
                Hg[i] = g * sl * B[i];
                dgp += sl * B[i] * __uint_as_float(ra[i]);
              } else {
                dA[i] = dH * ds;
                Hg[i] = g * sl;
                dgp += sl * __uint_as_float(ra[i]);
              }
            }
            staged_store<ER>(ring, &p.tmO0, t.n0 + 32 * c, wrow0, dA, valid, lane);
            if constexpr (SW) staged_store<ER>(ring, &p.tmO2, t.n0 + 32 * c, wrow0, dB, valid, lane);
            // Hg for the dW3 GEMM (not with MOEBLAZE_RECOMPUTE_H)
            if (p.o1) staged_store<ER>(ring, &p.tmO1, t.n0 + 32 * c, wrow0, Hg, valid, lane);
          }
          if (valid && p.dg) atomicAdd(p.dg + (int64_t)tok * p.K + kslot, dgp);
        }
      } else {
        // weight gradients: rows of dW_e, plain bf16 stores (wide tiles:
        // the second 128 rows from accumulator columns 256-511)
#pragma unroll 1
        for (int hm = 0; hm < (WIDE_T ? 2 : 1); ++hm) {
          if (WIDE_T && MODE == DW3_H && t.row0 + hm * BM >= p.h) break;  // half tile past the last row of dW3
          const int64_t orow = (int64_t)(t.row0 + hm * BM + r);
          const uint32_t tb = tbase + hm * 256;
          if constexpr (MODE == DW12) {
            const int64_t base = (int64_t)t.e * p.d * p.h + orow * p.h + t.n0;
            for (int c = 0; c < 8; ++c) {
              __nv_bfloat16* dst = (c < 4 ? p.o0 : p.o1) + base + 32 * (c & 3);
              if (t.kblocks > 0) {
                MB_TMEM_LD32(tb + 32 * c, ra);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) va[i] = __uint_as_float(ra[i]);
                store_row32(dst, va);
              } else {
                store_zero32(dst);
              }
            }
          } else {
            const int ld = MODE == DW1 ? p.h : p.d;
            const int64_t rows_e = MODE == DW1 ? p.d : p.h;
            const int64_t base = (int64_t)t.e * rows_e * ld + orow * ld + t.n0;
            for (int c = 0; c < t.nw / 32; ++c) {
              if (t.kblocks > 0) {
                MB_TMEM_LD32(tb + 32 * c, ra);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) va[i] = __uint_as_float(ra[i]);
                store_row32(p.o0 + base + 32 * c, va);
              } else {
                store_zero32(p.o0 + base + 32 * c);
              }
            }
          }
        }
      }
      (void)rb; (void)vb;
      tc_fence_before();
      mbar_arrive(bar(10 + abuf));
      if (++abuf == NACC) { abuf = 0; aph ^= 1u; }
    }
    // the TMA stores issued by lane 0 complete before the CTA exits
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // no multicast or remote arrive is still headed for this CTA
  tc_fence_after();
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
  }
}

// ------------------------------------------------------------------ host side
// Launch one GEMM stage.  `tiles_bound` bounds the number of 128-row tiles;
// one CTA per SM, never more than there are tiles.  PAIR: clusters of two
// CTAs on pairs of tiles (see the kernel).
template <int MODE, int VAR = SINGLE>
moeblaze_status launch(Params& p, int64_t tiles_bound, cudaStream_t st) {
  if (tiles_bound <= 0) return MOEBLAZE_OK;
  auto kern = moe_gemm_kernel<MODE, VAR>;
  constexpr int smem = smem_bytes_of(MODE, VAR);
  MB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  if constexpr (VAR == PAIRED) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * (sm_count() / 2)));
    cfg.blockDim = dim3(num_threads(MODE, VAR));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many clusters as can be resident at once, never more than pair tiles
    static int resident[64][16] = {};
    int dev = 0;
    MB_CUDA(cudaGetDevice(&dev));
    int& clusters = resident[dev & 63][MODE & 15];
    if (clusters == 0) {
      MB_CUDA(cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg));
      if (clusters < 1) return MOEBLAZE_ERR_UNSUPPORTED;
    }
    const int64_t pairs = tiles_bound / 2 < clusters ? tiles_bound / 2 : clusters;
    if (pairs < 1) return MOEBLAZE_OK;
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    MB_CUDA(cudaLaunchKernelEx(&cfg, kern, p));
  } else {
    const int64_t g = tiles_bound < sm_count() ? tiles_bound : sm_count();
    kern<<<(unsigned)g, num_threads(MODE, VAR), smem, st>>>(p);
  }
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

// MOEBLAZE_RECOMPUTE_H: the saved buffer is A | B (SwiGLU) | one fp32 gate per padded row
float* saved_row_gates(const __nv_bfloat16* saved, const moeblaze_shape& s) {
  const int64_t rows = max_padded_rows(s.L * s.K, s.E);
  const int nb = s.act == MOEBLAZE_SWIGLU ? 2 : 1;
  return reinterpret_cast<float*>(const_cast<__nv_bfloat16*>(saved) + (int64_t)nb * rows * s.h);
}

Params base_params(const moeblaze_shape& s, const moeblaze_dispatch& disp, const float* gates) {
  Params p;
  memset(&p, 0, sizeof(p));
  p.D1 = disp.expert_token_indices;
  p.D2 = disp.expert_token_offsets;
  p.D3 = disp.token_expert_indices;
  p.gates = gates;
  p.meta = meta_view(disp.meta, s.E);
  p.L = s.L;
  p.d = s.d; p.h = s.h; p.E = s.E; p.K = s.K;
  fault_injection(&p.wait_ns, &p.withhold);
  if (p.wait_ns == 0) p.wait_ns = kTimeoutNs;
  return p;
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    float4 v = src[i];
    dst[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

moeblaze_status convert(const float* src, __nv_bfloat16* dst, int64_t n, cudaStream_t st) {
  if (n == 0) return MOEBLAZE_OK;
  const int64_t n4 = n / 4;  // n = L*d with d % 128 == 0
  const int blocks = sm_count() * 8;
  f32_to_bf16_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(src), reinterpret_cast<uint2*>(dst), n4);
  MB_CUDA(cudaGetLastError());
  count_launch();
  return MOEBLAZE_OK;
}

}  // namespace tc

using namespace tc;

moeblaze_status tc_forward(const moeblaze_shape& s, const __nv_bfloat16* x, const float* gates,
                           const moeblaze_dispatch& disp, const __nv_bfloat16* W1, const __nv_bfloat16* W2,
                           const __nv_bfloat16* W3, __nv_bfloat16* y, __nv_bfloat16* saved, __nv_bfloat16* wsH,
                           float* wsY32, cudaStream_t st) {
  const bool sw = s.act == MOEBLAZE_SWIGLU;
  const bool rec = wsH == nullptr;  // MOEBLAZE_RECOMPUTE_H: no H temporary; the row gates are kept in saved
  const int64_t LK = s.L * s.K;
  const int64_t rows = max_padded_rows(LK, s.E);
  const int64_t mt_bound = rows / BM;
  // y32 and, behind it, the tile counters of the two launches start at zero
  const size_t y32_bytes = (sizeof(float) * s.L * s.d + 255) / 256 * 256;
  unsigned long long* sched = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(wsY32) + y32_bytes);
  MB_CUDA(cudaMemsetAsync(wsY32, 0, y32_bytes + kSchedBytes, st));
  stage_event(0, st);
  if (s.L > 0) {
    __nv_bfloat16* A = saved;
    __nv_bfloat16* B = sw ? saved + rows * s.h : nullptr;
    {  // up projection
      Params p = base_params(s, disp, gates);
      p.gsrc = x;
      p.gld = s.d;
      if (!make_map(&p.tmB0, W1, s.h, (uint64_t)s.E * s.d, 64, 64)) return MOEBLAZE_ERR_CUDA;
      if (sw && !make_map(&p.tmB1, W2, s.h, (uint64_t)s.E * s.d, 64, 64)) return MOEBLAZE_ERR_CUDA;
      p.N = s.h;
      p.kblocks = s.d / BK;
      p.ksplit = p.kblocks;
      p.n_tiles = (s.h + tile_n(sw ? UP_SWIGLU : UP_SILU) - 1) / tile_n(sw ? UP_SWIGLU : UP_SILU);
      p.o0 = A; p.o1 = B; p.o2 = wsH;
      p.sched = sched + 0;
      const CUtensorMapSwizzle s64 = CU_TENSOR_MAP_SWIZZLE_64B;
      if (!make_map(&p.tmO0, A, s.h, rows, 32, 32, s64)) return MOEBLAZE_ERR_CUDA;
      if (sw && !make_map(&p.tmO1, B, s.h, rows, 32, 32, s64)) return MOEBLAZE_ERR_CUDA;
      if (!rec && !make_map(&p.tmO2, wsH, s.h, rows, 32, 32, s64)) return MOEBLAZE_ERR_CUDA;
      // long reductions with many tiles: 256-row tiles (pairs of 128-row tiles of one expert)
      const int64_t nt = mt_bound * p.n_tiles;
      const bool wide = wide_rows(p.kblocks, nt);
      moeblaze_status r = sw ? (wide ? launch<UP_SWIGLU, WIDE>(p, nt / 2, st) : launch<UP_SWIGLU>(p, nt, st))
                             : (wide ? launch<UP_SILU, WIDE>(p, nt / 2, st) : launch<UP_SILU>(p, nt, st));
      if (r != MOEBLAZE_OK) return r;
    }
    stage_event(1, st);
    {  // down projection of H (stored, or recomputed from the saved tiles) + gate-weighted combine into y32
      Params p = base_params(s, disp, gates);
      if (!make_map(&p.tmA, rec ? A : wsH, s.h, rows, 64, 128)) return MOEBLAZE_ERR_CUDA;
      if (rec && sw && !make_map(&p.tmX, B, s.h, rows, 64, 128)) return MOEBLAZE_ERR_CUDA;
      if (!make_map(&p.tmB0, W3, s.d, (uint64_t)s.E * s.h, 64, 64)) return MOEBLAZE_ERR_CUDA;
      p.N = s.d;
      p.kblocks = s.h / BK;
      p.ksplit = p.kblocks;
      p.n_tiles = (s.d + 255) / 256;
      p.acc32 = wsY32;
      p.rowg = rec ? saved_row_gates(saved, s) : nullptr;
      p.sched = sched + 1;
      const int64_t nt = mt_bound * p.n_tiles;
      const bool wide = wide_rows(p.kblocks, nt);
      moeblaze_status r = !rec ? (wide ? launch<DOWN_H, WIDE>(p, nt / 2, st) : launch<DOWN_H>(p, nt, st))
                               : (sw ? launch<DOWN_SWIGLU>(p, nt, st) : launch<DOWN_SILU>(p, nt, st));
      if (r != MOEBLAZE_OK) return r;
    }
  }
  stage_event(2, st);
  moeblaze_status r = convert(wsY32, y, s.L * s.d, st);
  stage_event(3, st);
  return r;
}

moeblaze_status tc_backward(const moeblaze_shape& s, const __nv_bfloat16* dY, const __nv_bfloat16* x,
                            const float* gates, const moeblaze_dispatch& disp, const __nv_bfloat16* W1,
                            const __nv_bfloat16* W2, const __nv_bfloat16* W3, __nv_bfloat16* saved,
                            __nv_bfloat16* dX, __nv_bfloat16* dW1, __nv_bfloat16* dW2, __nv_bfloat16* dW3,
                            float* dgates, __nv_bfloat16* wsHg, float* wsdX32, cudaStream_t st) {
  // The saved A and B are read for the last time by the dH GEMM, which reads
  // and writes the same (row, column) positions, so its dA and dB overwrite
  // them in place and the dX and dW1|dW2 GEMMs read them from there.
  // Default: dH also stores Hg (scratch) for the dW3 GEMM, which runs last.
  // MOEBLAZE_RECOMPUTE_H (wsHg NULL): dW3 runs first, recomputing
  // Hg = g SiLU(A) B from the saved A, B and the row gates the forward kept.
  const bool rec = wsHg == nullptr;
  const bool sw = s.act == MOEBLAZE_SWIGLU;
  const int64_t LK = s.L * s.K;
  const int64_t rows = max_padded_rows(LK, s.E);
  const int64_t mt_bound = rows / BM;
  __nv_bfloat16* A = saved;                                  // A, then dA
  __nv_bfloat16* B = sw ? saved + rows * s.h : nullptr;      // B, then dB
  // dX32 and, behind it, the tile counters of the four launches start at zero
  const size_t dx32_bytes = (sizeof(float) * s.L * s.d + 255) / 256 * 256;
  unsigned long long* sched = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(wsdX32) + dx32_bytes);
  MB_CUDA(cudaMemsetAsync(wsdX32, 0, dx32_bytes + kSchedBytes, st));
  int ev = 0;
  stage_event(ev++, st);
  auto dw3 = [&]() -> moeblaze_status {  // dW3 = Hg^T dY
    Params p = base_params(s, disp, gates);
    if (!make_map(&p.tmA, rec ? A : wsHg, s.h, rows, 64, 64)) return MOEBLAZE_ERR_CUDA;
    if (rec && sw && !make_map(&p.tmX, B, s.h, rows, 64, 64)) return MOEBLAZE_ERR_CUDA;
    p.rowg = rec ? saved_row_gates(saved, s) : nullptr;
    p.gsrc = dY;
    p.gld = s.d;
    p.N = s.d;
    const bool wide = !rec && wide_stage(s, s.h, true);
    p.m_tiles_w = wide ? (s.h + 2 * BM - 1) / (2 * BM) : s.h / BM;
    p.n_tiles = (s.d + 255) / 256;
    p.total_w = (int64_t)s.E * p.m_tiles_w * p.n_tiles;
    p.o0 = dW3;
    p.sched = sched + 3;
    moeblaze_status r = rec    ? (sw ? launch<DW3_SWIGLU>(p, p.total_w, st) : launch<DW3_SILU>(p, p.total_w, st))
                        : wide ? launch<DW3_H, WIDE>(p, p.total_w, st)
                               : launch<DW3_H>(p, p.total_w, st);
    if (r == MOEBLAZE_OK) stage_event(ev++, st);
    return r;
  };
  if (rec) {
    moeblaze_status r = dw3();
    if (r != MOEBLAZE_OK) return r;
  }
  {  // dH = dY W3^T with the SwiGLU backward epilogue; dA, dB over A, B
    Params p = base_params(s, disp, gates);
    p.gsrc = dY;
    p.gld = s.d;
    if (!make_map(&p.tmB0, W3, s.d, (uint64_t)s.E * s.h, 64, 128)) return MOEBLAZE_ERR_CUDA;
    p.N = s.h;
    p.kblocks = s.d / BK;
    p.ksplit = p.kblocks;
    p.n_tiles = (s.h + 255) / 256;
    p.o1 = wsHg; p.i0 = A; p.i1 = B;
    p.dg = dgates;
    p.sched = sched + 0;
    const CUtensorMapSwizzle s64 = CU_TENSOR_MAP_SWIZZLE_64B;
    if (!make_map(&p.tmO0, A, s.h, rows, 32, 32, s64)) return MOEBLAZE_ERR_CUDA;
    if (sw && !make_map(&p.tmO2, B, s.h, rows, 32, 32, s64)) return MOEBLAZE_ERR_CUDA;
    if (!rec && !make_map(&p.tmO1, wsHg, s.h, rows, 32, 32, s64)) return MOEBLAZE_ERR_CUDA;
    const int64_t nt = mt_bound * p.n_tiles;
    const bool pair = pair_stage(p.kblocks, nt);
    moeblaze_status r = sw ? (pair ? launch<DH_SWIGLU, PAIRED>(p, nt, st) : launch<DH_SWIGLU>(p, nt, st))
                           : (pair ? launch<DH_SILU, PAIRED>(p, nt, st) : launch<DH_SILU>(p, nt, st));
    if (r != MOEBLAZE_OK) return r;
  }
  stage_event(ev++, st);
  {  // dX = dA W1^T + dB W2^T, reduced into dX32
    Params p = base_params(s, disp, gates);
    if (!make_map(&p.tmA, A, s.h, rows, 64, 128)) return MOEBLAZE_ERR_CUDA;
    if (sw && !make_map(&p.tmX, B, s.h, rows, 64, 128)) return MOEBLAZE_ERR_CUDA;
    if (!make_map(&p.tmB0, W1, s.h, (uint64_t)s.E * s.d, 64, 128)) return MOEBLAZE_ERR_CUDA;
    if (sw && !make_map(&p.tmB1, W2, s.h, (uint64_t)s.E * s.d, 64, 128)) return MOEBLAZE_ERR_CUDA;
    p.N = s.d;
    p.kblocks = (sw ? 2 : 1) * s.h / BK;
    p.ksplit = s.h / BK;
    p.n_tiles = (s.d + 255) / 256;
    p.acc32 = wsdX32;
    p.sched = sched + 1;
    const int64_t nt = mt_bound * p.n_tiles;
    moeblaze_status r = wide_rows(p.kblocks, nt) ? launch<DX, WIDE>(p, nt / 2, st) : launch<DX>(p, nt, st);
    if (r != MOEBLAZE_OK) return r;
  }
  stage_event(ev++, st);
  {  // dW1 (and dW2) = X_e^T [dA | dB]
    Params p = base_params(s, disp, gates);
    p.gsrc = x;
    p.gld = s.d;
    if (!make_map(&p.tmB0, A, s.h, rows, 64, 64)) return MOEBLAZE_ERR_CUDA;
    if (sw && !make_map(&p.tmB1, B, s.h, rows, 64, 64)) return MOEBLAZE_ERR_CUDA;
    p.N = s.h;
    const bool wide = wide_stage(s, s.d, false);
    p.m_tiles_w = s.d / (wide ? 2 * BM : BM);
    p.n_tiles = sw ? s.h / 128 : (s.h + 255) / 256;
    p.total_w = (int64_t)s.E * p.m_tiles_w * p.n_tiles;
    p.o0 = dW1; p.o1 = dW2;
    p.sched = sched + 2;
    moeblaze_status r = sw ? (wide ? launch<DW12, WIDE>(p, p.total_w, st) : launch<DW12>(p, p.total_w, st))
                           : (wide ? launch<DW1, WIDE>(p, p.total_w, st) : launch<DW1>(p, p.total_w, st));
    if (r != MOEBLAZE_OK) return r;
  }
  stage_event(ev++, st);
  if (!rec) {
    moeblaze_status r = dw3();
    if (r != MOEBLAZE_OK) return r;
  }
  moeblaze_status r = convert(wsdX32, dX, s.L * s.d, st);
  stage_event(ev++, st);
  return r;
}

}  // namespace moeblaze
