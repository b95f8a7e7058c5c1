// Tree attention on the 5th-generation tensor cores (bf16, head dim 128),
// flash-style ("Medusa Heads", "Attenzione sull'albero e accettazione": every
// candidate in one pass, each seeing the cache and its own ancestors).
//
//   o[b][i][h] = sum_j softmax_j(q . k_j / sqrt(Dh)) v_j
//   over cache rows j < L, then tree nodes j set in node i's ancestor mask.
//
// A CTA owns up to 256 query rows of one (sequence b, kv head g) as two
// 128-row tiles (row r is (node r / G, q head g*G + r % G), one TMEM lane of
// its tile each); both tiles share every K/V block, which streams in blocks
// of 64 keys (cache blocks, then tree blocks) through 3-deep K and V TMA
// rings.  The 4-D tensor maps give the key axis the extent L (or T), so rows
// past the valid keys read as zeros.  Per block and tile:
//   S = Q K^T     tcgen05.mma M=128, N=64, K=128 into one of two TMEM buffers
//                 of the tile (block i+1's product runs during block i's
//                 softmax)
//   softmax       4 warps per tile, one thread per row (64 scores): masked,
//                 scaled row max, P = exp2(s - m) packed to bf16 into the
//                 tile's 128-byte-swizzled P tile.  The running max is only
//                 raised (and O rescaled in TMEM) when it grows by more than
//                 2^8, so one m serves P, the row sum and the final division.
//                 The two tiles' softmax chains are independent and hide each
//                 other's latency.
//   O += P V      tcgen05.mma with V as an MN-major operand (the [key][dh]
//                 tile the TMA wrote), O resident in TMEM for the whole pass.
// Warp roles (one thread each for the first four, so no issue order couples
// loads or MMAs that do not depend on one another): warp 0 loads K, warp 1
// loads V, warp 2 allocates TMEM and issues S = Q K^T, warp 3 issues O += P V,
// warps 4..7 and 8..11 run the softmax and epilogue of tiles 0 and 1.  With
// fewer (row pair, b, g) CTAs than SMs the key blocks are split into NS equal
// shares (partials merged by the combine kernel).  In the fused step's overlap
// schedule the kernel runs unsplit beside the head projection, on the SMs the
// projection's grid leaves free.  Every wait is bounded.
#include <limits.h>

#include "internal.cuh"
#include "tc.cuh"

namespace medusa {

constexpr int AT_M = 128;            // query rows per tile
constexpr int AT_TILES = 2;          // tiles per CTA
constexpr int AT_ROWS = AT_M * AT_TILES;
constexpr int AT_BK = 64;            // keys per block
constexpr int AT_DH = 128;
constexpr int AT_STAGES = 4;         // depth of the K ring and of the V ring
constexpr int AT_THREADS = 128 + 32 * 4 * AT_TILES;
constexpr uint32_t AT_QCHUNK = AT_M * 128;        // 16 KB: 128 rows x 64 columns, 128-byte swizzled
constexpr uint32_t AT_QTILE = 2 * AT_QCHUNK;      // Q of a tile: [128 rows][128 dh]
constexpr uint32_t AT_KVCHUNK = AT_BK * 128;      // 8 KB: 64 keys x 64 dh
constexpr uint32_t AT_KVTILE = 2 * AT_KVCHUNK;    // K or V: [64 keys][128 dh]
constexpr uint32_t AT_TMEM_COLS = 512;            // per tile: S0, S1 (64 columns each; P over the first 32); then O of each tile (128)
constexpr uint64_t AT_WAIT_NS = 20ull * 1000 * 1000;
constexpr uint32_t AT_SLEEP_NS = 1000 * 1000;     // a waiting thread sleeps until its phase completes (<= 1 ms per poll)
constexpr float AT_RESCALE_LOG2 = 8.f;            // raise the running max only past 2^8 growth

struct AtArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  TreeDims td;
  int B, T, W, Hq, Hkv, G, L, H;
  int NS;
  float* part_o;
  float2* part_ml;
  float qscale;  // log2(e) / sqrt(Dh)
  uint8_t* ws;
  const int32_t* lens;  // [B] per-sequence cache lengths, or null (L for all)
  int Lc;
  // overlap schedule of the fused step: launched right after the head
  // projection, whose kernel lets it start only after everything before the
  // step has completed, so no store waits and the CTAs retire freely; each
  // CTA counts itself into *done_count once its outputs are written (the
  // verification projection waits for that count, not for this grid)
  int nowait;
  int* done_count;
};

__device__ __forceinline__ uint32_t at_sw(int r, int unit) {  // byte offset of 16-byte unit `unit` of row r
  return (uint32_t)((unit >> 3) * AT_QCHUNK + r * 128 + (((unit & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ bool at_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint8_t* ws) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::globaltimer_ns();
  while (!tc::mbar_try_wait_sleep(bar, parity, AT_SLEEP_NS)) {
    if (*abort_flag) return false;
    if (tc::globaltimer_ns() - t0 > AT_WAIT_NS) {
      set_error(ws, MEDUSA_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// one lane waits, the warp learns the verdict (the shuffle orders the other
// lanes after lane 0's observation of the phase)
__device__ __forceinline__ bool at_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint8_t* ws,
                                             int lane) {
  int okv = 0;
  if (lane == 0) okv = at_wait(bar, parity, abort_flag, ws) ? 1 : 0;
  return __shfl_sync(0xffffffffu, okv, 0) != 0;
}

// 2^x on the special-function unit (relative error ~2^-22; 2^-inf = 0;
// results below the normal range flush to zero, far below what a bf16
// probability resolves)
__device__ __forceinline__ float at_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float at_max3(float x, float y, float z) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(x), "f"(y), "f"(z));
  return d;
}

// (y0, y1) = (x0, x1) * s + c as one paired fp32 FMA (each lane rounds like fmaf)
__device__ __forceinline__ void at_fma2(float& y0, float& y1, float x0, float x1, float s, float c) {
  uint64_t x, sv, cv, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(sv) : "f"(s), "f"(s));
  asm("mov.b64 %0, {%1, %2};" : "=l"(cv) : "f"(c), "f"(c));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y) : "l"(x), "l"(sv), "l"(cv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(y0), "=f"(y1) : "l"(y));
}

// (a0, a1) += (x0, x1) as one paired fp32 add
__device__ __forceinline__ void at_add2(float& a0, float& a1, float x0, float x1) {
  uint64_t av, xv;
  asm("mov.b64 %0, {%1, %2};" : "=l"(av) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(xv) : "f"(x0), "f"(x1));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(av) : "l"(xv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(av));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmVc,
                        const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmVt,
                        const __grid_constant__ AtArgs a) {
  extern __shared__ uint8_t at_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Qs = smem;                                   // [tile] Q tiles
  uint8_t* Ks = Qs + AT_TILES * AT_QTILE;               // [AT_STAGES] K tiles
  uint8_t* Vs = Ks + AT_STAGES * AT_KVTILE;             // [AT_STAGES] V tiles
  uint32_t* mrow = reinterpret_cast<uint32_t*>(Vs + AT_STAGES * AT_KVTILE);  // [256][W] ancestor masks
  uint64_t* bars = reinterpret_cast<uint64_t*>(mrow + AT_ROWS * a.W);       // 256 * W words: 8-byte aligned
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + AT_STAGES;
  uint64_t* v_full = k_empty + AT_STAGES;
  uint64_t* v_empty = v_full + AT_STAGES;
  uint64_t* s_full = v_empty + AT_STAGES;    // [tile][2]
  uint64_t* s_free = s_full + 2 * AT_TILES;  // [tile][2]: the buffer's P V is done
  // [tile][block parity]: P(i) written by the tile's 4 warps.  A warp can be
  // at most one block ahead of another (block i + 1 needs S(i + 1), whose
  // buffer frees only after P(i - 1) V), so two barriers keep arrivals of
  // neighbouring blocks apart.
  uint64_t* p_full = s_free + 2 * AT_TILES;
  // [tile][block parity]: P(i) V complete.  Split by parity for the same
  // reason: a parity wait must never be more than one phase from its target.
  uint64_t* pv_done = p_full + 2 * AT_TILES;
  uint64_t* q_ready = pv_done + 2 * AT_TILES;
  uint64_t* drain = q_ready + 1;             // [2]: S issuer, PV issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y / a.NS, sp = blockIdx.y - g * a.NS, b = blockIdx.z;
  const int nrows = a.T * a.G;
  const int row0 = blockIdx.x * AT_ROWS;
  const int ntiles = min(AT_TILES, (nrows - row0 + AT_M - 1) / AT_M);
  const int Lb = seq_len(a.lens, b, a.L, a.Lc, a.ws);
  const int nb_cache = (Lb + AT_BK - 1) / AT_BK;
  const int nb_all = nb_cache + (a.T + AT_BK - 1) / AT_BK;
  const int blk_lo = (int)(((long long)sp * nb_all) / a.NS);
  const int blk_hi = (int)(((long long)(sp + 1) * nb_all) / a.NS);
  const int nblk = blk_hi - blk_lo;

  if (threadIdx.x == 0) {
    for (int s = 0; s < AT_STAGES; ++s) {
      tc::mbar_init(&k_full[s], 1);
      tc::mbar_init(&k_empty[s], 1);
      tc::mbar_init(&v_full[s], 1);
      tc::mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < AT_TILES; ++t) {
      for (int u = 0; u < 2; ++u) {
        tc::mbar_init(&s_full[2 * t + u], 1);
        tc::mbar_init(&s_free[2 * t + u], 1);
      }
      tc::mbar_init(&p_full[2 * t], 4);
      tc::mbar_init(&p_full[2 * t + 1], 4);
      tc::mbar_init(&pv_done[2 * t], 1);
      tc::mbar_init(&pv_done[2 * t + 1], 1);
    }
    tc::mbar_init(q_ready, 4 * AT_TILES);
    tc::mbar_init(&drain[0], 1);
    tc::mbar_init(&drain[1], 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmKc);
    tc::prefetch_tmap(&tmVc);
    tc::prefetch_tmap(&tmKt);
    tc::prefetch_tmap(&tmVt);
  }
  if (warp == 2) {
    tc::tmem_alloc(tmem_slot, AT_TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp <= 1) {
    // ------------------------------------------------- producers (K: warp 0, V: warp 1)
    // K(i) waits only for the S products of block i - 3, V(i) for its P V
    if (lane == 0) {
      const bool isv = warp == 1;
      uint64_t* full = isv ? v_full : k_full;
      uint64_t* empty = isv ? v_empty : k_empty;
      uint8_t* base = isv ? Vs : Ks;
      int n = 0;
      for (; n < nblk; ++n) {
        const int s = n % AT_STAGES;
        if (!at_wait(&empty[s], ((n / AT_STAGES) & 1u) ^ 1u, abort_flag, a.ws)) break;
        const int blk = blk_lo + n;
        const bool tree = blk >= nb_cache;
        const int k0 = tree ? (blk - nb_cache) * AT_BK : blk * AT_BK;
        const CUtensorMap* map = isv ? (tree ? &tmVt : &tmVc) : (tree ? &tmKt : &tmKc);
        tc::mbar_arrive_expect_tx(&full[s], AT_KVTILE);
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tc::tma_load_4d(base + (size_t)s * AT_KVTILE + c * AT_KVCHUNK, map, &full[s], c * 64, g, k0, b);
      }
      if (n < nblk) {  // aborted: drain the copies already issued
        for (int j = (n > AT_STAGES ? n - AT_STAGES : 0); j < n; ++j) {
          const uint64_t t0 = tc::globaltimer_ns();
          while (!tc::mbar_try_wait(&full[j % AT_STAGES], (j / AT_STAGES) & 1u) &&
                 tc::globaltimer_ns() - t0 < AT_WAIT_NS) {
          }
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------- S = Q K^T issue
    if (lane == 0) {
      const uint32_t idS = tc::idesc_bf16_f32(AT_M, AT_BK);
      bool ok = at_wait(q_ready, 0, abort_flag, a.ws);
      for (int i = 0; i < nblk && ok; ++i) {
        const int s = i % AT_STAGES, buf = i & 1;
        if (!at_wait(&k_full[s], (i / AT_STAGES) & 1u, abort_flag, a.ws)) {
          ok = false;
          break;
        }
        const uint32_t ka = tc::smem_u32(Ks + (size_t)s * AT_KVTILE);
        for (int t = 0; t < ntiles && ok; ++t) {  // S(t, i) into TMEM buffer i % 2 of tile t
          if (!at_wait(&s_free[2 * t + buf], ((i >> 1) & 1u) ^ 1u, abort_flag, a.ws)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t qa = tc::smem_u32(Qs + t * AT_QTILE);
#pragma unroll
          for (int c = 0; c < 2; ++c)  // dh chunks
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_bf16(tmem + t * 2 * AT_BK + buf * AT_BK, tc::sw128_desc(qa + c * AT_QCHUNK) + 2 * kk,
                           tc::sw128_desc(ka + c * AT_KVCHUNK) + 2 * kk, idS, (c | kk) != 0);
          tc::mma_commit(&s_full[2 * t + buf]);
        }
        if (ok) tc::mma_commit(&k_empty[s]);
      }
      tc::mma_commit(&drain[0]);  // every MMA of this thread completes before TMEM is freed
      const uint64_t t0 = tc::globaltimer_ns();
      while (!tc::mbar_try_wait(&drain[0], 0) && tc::globaltimer_ns() - t0 < AT_WAIT_NS) {
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------- O += P V issue
    if (lane == 0) {
      const uint32_t idO = tc::idesc_bf16_f32(AT_M, AT_DH) | (1u << 16);  // V: MN-major B operand
      bool ok = true;
      for (int i = 0; i < nblk && ok; ++i) {
        const int s = i % AT_STAGES;
        if (!at_wait(&v_full[s], (i / AT_STAGES) & 1u, abort_flag, a.ws)) {
          ok = false;
          break;
        }
        const uint32_t va = tc::smem_u32(Vs + (size_t)s * AT_KVTILE);
        for (int t = 0; t < ntiles && ok; ++t) {
          if (!at_wait(&p_full[2 * t + (i & 1)], (i >> 1) & 1u, abort_flag, a.ws)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t pt = tmem + t * 2 * AT_BK + (i & 1) * AT_BK;  // P(i): bf16 pairs over S(i)
#pragma unroll
          for (int st = 0; st < AT_BK / 16; ++st) {  // 16 keys per MMA: 8 TMEM columns of A
            uint64_t db = tc::sw128_desc(va + st * 2048);
            db = (db & ~(0x3FFFull << 16)) | ((uint64_t)(AT_KVCHUNK >> 4) << 16);  // dh-chunk stride
            tc::mma_bf16_tmem_a(tmem + AT_TILES * 2 * AT_BK + t * AT_DH, pt + st * 8, db, idO, (i | st) != 0);
          }
          tc::mma_commit(&pv_done[2 * t + (i & 1)]);
          tc::mma_commit(&s_free[2 * t + (i & 1)]);  // the S buffer held P(i)
        }
        if (ok) tc::mma_commit(&v_empty[s]);
      }
      tc::mma_commit(&drain[1]);
      const uint64_t t0 = tc::globaltimer_ns();
      while (!tc::mbar_try_wait(&drain[1], 0) && tc::globaltimer_ns() - t0 < AT_WAIT_NS) {
      }
    }
  } else {
    // ------------------------------------------------- softmax of tile t
    const int t = (warp - 4) >> 2;
    const int q4 = warp & 3;                       // TMEM lane quadrant (warps 4..7 and 8..11 take 0..3)
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int trow = q4 * 32 + lane;               // row within the tile = TMEM lane
    const int r = row0 + t * AT_M + trow;          // query row
    const bool rvalid = r < nrows;
    const int node = rvalid ? r / a.G : 0;
    const int hq = g * a.G + (rvalid ? r - node * a.G : 0);
    uint8_t* Qt = Qs + t * AT_QTILE;
    // Q row into the swizzled tile (zeros for padding rows)
    {
      const uint4* src = reinterpret_cast<const uint4*>(a.q + (((size_t)b * a.T + node) * a.Hq + hq) * AT_DH);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint4 v = rvalid ? src[u] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(Qt + at_sw(trow, u)) = v;
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(q_ready);
    }
    // ancestor-or-self mask of this row's node (the chain of parents)
    uint32_t* mr = mrow + (size_t)(t * AT_M + trow) * a.W;
    for (int w = 0; w < a.W; ++w) mr[w] = 0u;
    if (rvalid)
      for (int j = node; j >= 0; j = a.td.parent[j]) mr[j >> 5] |= 1u << (j & 31);
    const bool warp_live = t < ntiles && (row0 + t * AT_M + q4 * 32) < nrows;  // some row of this warp is real
    const bool tile_live = t < ntiles;
    const uint32_t sbase = tmem + lane_off + t * 2 * AT_BK;
    const uint32_t obase = tmem + lane_off + AT_TILES * 2 * AT_BK + t * AT_DH;
    float m = -INFINITY, l = 0.f;
    bool ok = tile_live;
    for (int i = 0; i < nblk && ok; ++i) {
      const int buf = i & 1;
      const int blk = blk_lo + i;
      const bool tree = blk >= nb_cache;
      const int k0 = tree ? (blk - nb_cache) * AT_BK : blk * AT_BK;
      const int nk = tree ? min(AT_BK, a.T - k0) : min(AT_BK, Lb - k0);
      uint32_t mw0 = 0u, mw1 = 0u;  // mask words of the block's 64 keys
      if (tree) {
        const int wi = k0 >> 5;
        mw0 = wi < a.W ? mr[wi] : 0u;
        mw1 = wi + 1 < a.W ? mr[wi + 1] : 0u;
      }
      if (!at_wait_warp(&s_full[2 * t + buf], (i >> 1) & 1u, abort_flag, a.ws, lane)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // the row's 64 scores into registers; the S buffer is released at once
      float v[AT_BK];
      if (warp_live) {
        float(&va)[32] = *reinterpret_cast<float(*)[32]>(&v[0]);
        float(&vb)[32] = *reinterpret_cast<float(*)[32]>(&v[32]);
        const uint32_t sb = sbase + buf * AT_BK;
        tc::tmem_ld32_nowait(sb, va);
        tc::tmem_ld32_nowait(sb + 32, vb);
        tc::tmem_wait_ld();
        tc::tmem_regs_ready32(va);
        tc::tmem_regs_ready32(vb);
      }
      if (!warp_live) {  // no real row: nothing to compute, the handshake goes on
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&p_full[2 * t + buf]);
        continue;
      }
      // a full cache block needs no visibility test; elsewhere a hidden key
      // gets -inf (branch-free loops, the test sits outside them)
      const bool plain = !tree && nk >= AT_BK;
      if (!plain) {
#pragma unroll
        for (int kk = 0; kk < AT_BK; ++kk) {
          bool vis = rvalid && kk < nk;
          if (tree) vis = vis && (((kk < 32 ? mw0 : mw1) >> (kk & 31)) & 1u);
          v[kk] = vis ? v[kk] : -INFINITY;
        }
      }
      // row max of the block: a tree of three-input maxima (21 + 7 + 4)
      static_assert(AT_BK == 64, "the max tree below is written for 64 keys");
      float m1[22], m2[8];
#pragma unroll
      for (int j = 0; j < 21; ++j) m1[j] = at_max3(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
      m1[21] = v[63];
#pragma unroll
      for (int j = 0; j < 7; ++j) m2[j] = at_max3(m1[3 * j], m1[3 * j + 1], m1[3 * j + 2]);
      m2[7] = m1[21];
      const float bmax = at_max3(at_max3(m2[0], m2[1], m2[2]), at_max3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7]));
      const float mx = bmax * a.qscale;  // the scale is positive; -inf stays -inf
      {
        const bool raise = mx > m + AT_RESCALE_LOG2 || (m == -INFINITY && mx > -INFINITY);
        const float mn = raise ? mx : m;
        const bool resc = raise && i > 0 && m > -INFINITY;
        const float sc = resc ? exp2f(m - mn) : 1.f;
        if (resc) l *= sc;
        if (__any_sync(0xffffffffu, resc)) {  // rescale the accumulated O rows in TMEM (whole warp)
          // after P(i-1) V has landed in O
          if (!at_wait_warp(&pv_done[2 * t + ((i - 1) & 1)], ((i - 1) >> 1) & 1u, abort_flag, a.ws, lane)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < AT_DH / 16; ++c) {
            float o[16];
            tc::tmem_ld16(obase + c * 16, o);
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] *= sc;
            tc::tmem_st16(obase + c * 16, o);
          }
          tc::tmem_wait_st();
        }
        m = mn;
      }
      // P = exp2(s * scale - m) (a -inf score gives 0) as bf16 pairs (the
      // even key in the low half) over the first 32 columns of S(i) in TMEM
      const float nm = (m == -INFINITY) ? 0.f : -m;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      uint32_t pk[AT_BK / 2];
#pragma unroll
      for (int j = 0; j < AT_BK; j += 4) {  // paired FMAs and adds around the exponentials
        float x0, x1, x2, x3;
        at_fma2(x0, x1, v[j], v[j + 1], a.qscale, nm);
        at_fma2(x2, x3, v[j + 2], v[j + 3], a.qscale, nm);
        const float p0 = at_exp2(x0), p1 = at_exp2(x1), p2 = at_exp2(x2), p3 = at_exp2(x3);
        at_add2(s0, s1, p0, p1);
        at_add2(s2, s3, p2, p3);
        pk[j >> 1] = pack2_bf16(p0, p1);
        pk[(j >> 1) + 1] = pack2_bf16(p2, p3);
      }
      tc::tmem_st32_nowait(sbase + buf * AT_BK, pk);
      tc::tmem_wait_st();
      l += (s0 + s1) + (s2 + s3);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&p_full[2 * t + buf]);
    }
    // ---- epilogue: wait for the last P V, then O / l (or the partial).  The
    // stores wait for the preceding grid (the previous step may still read
    // the output); everything above reads only this step's inputs.
    if (ok && nblk > 0 &&
        !at_wait_warp(&pv_done[2 * t + ((nblk - 1) & 1)], ((nblk - 1) >> 1) & 1u, abort_flag, a.ws, lane))
      ok = false;
    if (!a.nowait) pdl_wait();
    tc::fence_after_sync();
    if (ok && warp_live && nblk > 0) {  // TMEM loads by the whole warp, stores by the real rows
      if (a.NS > 1) {
        const size_t pr = (((size_t)b * a.Hq + hq) * a.T + node) * a.NS + sp;
        float* po = a.part_o + pr * AT_DH;
#pragma unroll
        for (int c = 0; c < AT_DH / 16; ++c) {
          float o[16];
          tc::tmem_ld16(obase + c * 16, o);
          if (rvalid)
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(po + c * 16 + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
        }
        if (rvalid) a.part_ml[pr] = make_float2(m, l);
      } else {
        const float inv = rvalid ? 1.f / l : 0.f;
        __nv_bfloat16* op = a.out + ((size_t)b * a.T + node) * a.H + (size_t)hq * AT_DH;
#pragma unroll
        for (int c = 0; c < AT_DH / 16; ++c) {
          float o[16];
          tc::tmem_ld16(obase + c * 16, o);
          if (!rvalid) continue;
          uint4 w0, w1;
          w0.x = pack2_bf16(o[0] * inv, o[1] * inv);
          w0.y = pack2_bf16(o[2] * inv, o[3] * inv);
          w0.z = pack2_bf16(o[4] * inv, o[5] * inv);
          w0.w = pack2_bf16(o[6] * inv, o[7] * inv);
          w1.x = pack2_bf16(o[8] * inv, o[9] * inv);
          w1.y = pack2_bf16(o[10] * inv, o[11] * inv);
          w1.z = pack2_bf16(o[12] * inv, o[13] * inv);
          w1.w = pack2_bf16(o[14] * inv, o[15] * inv);
          *reinterpret_cast<uint4*>(op + c * 16) = w0;
          *reinterpret_cast<uint4*>(op + c * 16 + 8) = w1;
        }
      }
    } else if (ok && warp_live && nblk == 0 && a.NS > 1 && rvalid) {  // a split with no key block
      a.part_ml[(((size_t)b * a.Hq + hq) * a.T + node) * a.NS + sp] = make_float2(-INFINITY, 0.f);
    } else if (!ok && tile_live && lane == 0) {
      set_error(a.ws, MEDUSA_ERR_TIMEOUT);
    }
  }

  // ---------------------------------------------------------------- teardown
  if (a.done_count) __threadfence();  // this thread's outputs, before the count below
  tc::fence_before_sync();
  __syncthreads();
  if (a.done_count && threadIdx.x == 0) atomicAdd(a.done_count, 1);
  if (warp == 2) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, AT_TMEM_COLS);
  }
  if (!a.nowait) pdl_wait();  // completes only after the preceding kernel (keeps the stream's order transitive)
}

// ------------------------------------------------------------------- host --
typedef CUresult (*AtEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static AtEncodeFn at_encode_fn() {
  static AtEncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<AtEncodeFn>(p);
  }
  return fn;
}

// [B][rows_alloc][Hkv][128] bf16 viewed as (dh, kv head, key < rows, sequence):
// box (64, 1, 128, 1); keys at or past `rows` read as zero.
static int at_kv_map(CUtensorMap* m, const void* base, int B, int rows, int rows_alloc, int Hkv) {
  AtEncodeFn fn = at_encode_fn();
  if (!fn) return (int)cudaErrorNotSupported;
  cuuint64_t dims[4] = {(cuuint64_t)AT_DH, (cuuint64_t)Hkv, (cuuint64_t)rows, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)AT_DH * 2, (cuuint64_t)Hkv * AT_DH * 2,
                           (cuuint64_t)rows_alloc * Hkv * AT_DH * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)AT_BK, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

// Key splits: when the (256-row pair, b, kv head) CTAs do not fill the ~148
// SMs, their key blocks are cut into NS equal shares, NS chosen for the
// shortest last wave (device independent, so the workspace can be sized from
// the config alone).  A full grid is never split: the partials would cost
// more traffic than the tail they save.
int attn_tc_splits(int B, int T, int G, int Hkv, int L) {
  constexpr int kSlots = 148;
  if (L == 0) return 1;
  const long long units = (long long)((T * G + AT_ROWS - 1) / AT_ROWS) * Hkv * B;
  if (units >= kSlots) return 1;
  const int nb_all = (L + AT_BK - 1) / AT_BK + (T + AT_BK - 1) / AT_BK;
  int best = 1;
  double best_cost = 1e30;
  for (int ns = 1; ns <= 8 && ns <= nb_all / 2 + (ns == 1); ++ns) {
    const long long waves = (units * ns + kSlots - 1) / kSlots;
    const double cost = (double)waves / ns + 0.03 * (ns - 1);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = ns;
    }
  }
  return best;
}

bool attn_tc_supported(const Plan& p) { return p.bf16 && p.Dh == AT_DH; }

long long attn_tc_unsplit_ctas(const Plan& p) {
  return (long long)((p.T * p.G + AT_ROWS - 1) / AT_ROWS) * p.Hkv * p.B;
}

int launch_attn_combine(const Plan& p, float* part_o, float2* part_ml, int NS, void* out, cudaStream_t st);

int launch_tree_attn_tc(const Plan& p, const void* q, const void* kt, const void* vt, const void* kc, const void* vc,
                        const int32_t* lens, void* out, uint8_t* ws, cudaStream_t st) {
  AtArgs a;
  a.q = (const __nv_bfloat16*)q;
  a.out = (__nv_bfloat16*)out;
  a.td = p.tree;
  a.B = p.B;
  a.T = p.T;
  a.W = p.W;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.G = p.G;
  a.L = p.L;
  a.H = p.H;
  a.qscale = 1.4426950408889634f / sqrtf((float)p.Dh);
  a.ws = ws;
  a.lens = lens;
  a.Lc = p.Lc;
  // beside the projection the attention has only the SMs the projection
  // leaves free: no key splits (and no combine launch)
  a.NS = p.overlap ? 1 : attn_tc_splits(p.B, p.T, p.G, p.Hkv, p.L);
  a.nowait = p.overlap ? 1 : 0;
  a.done_count = p.overlap ? reinterpret_cast<int*>(ws) + TICKET_ATTN_DONE : nullptr;
  const size_t rows_all = (size_t)p.B * p.Hq * p.T * a.NS;
  a.part_o = reinterpret_cast<float*>(ws + p.off_attn_part);
  a.part_ml = reinterpret_cast<float2*>(ws + p.off_attn_part + rows_all * p.Dh * sizeof(float));
  CUtensorMap mkt, mvt, mkc, mvc;
  int e = at_kv_map(&mkt, kt, p.B, p.T, p.T, p.Hkv);
  if (!e) e = at_kv_map(&mvt, vt, p.B, p.T, p.T, p.Hkv);
  // key extent: L, or the capacity when each sequence has its own length
  // (rows past a sequence's length are masked as keys and weighted 0 as values)
  const int ext = lens ? p.Lc : p.L;
  if (!e && ext > 0) e = at_kv_map(&mkc, kc, p.B, ext, p.Lc, p.Hkv);
  if (!e && ext > 0) e = at_kv_map(&mvc, vc, p.B, ext, p.Lc, p.Hkv);
  if (e) return e;
  if (ext == 0) {  // no cache blocks exist: the cache maps are never used
    mkc = mkt;
    mvc = mvt;
  }
  const size_t smem = 1024 + (size_t)AT_TILES * AT_QTILE + (size_t)2 * AT_STAGES * AT_KVTILE +
                      (size_t)AT_ROWS * p.W * sizeof(uint32_t) + 512;
  cudaError_t ce = cudaFuncSetAttribute(tree_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (ce != cudaSuccess) return (int)ce;
  dim3 grid((p.T * p.G + AT_ROWS - 1) / AT_ROWS, p.Hkv * a.NS, p.B);
  // programmatic dependent launch: the pass runs beside the preceding kernels,
  // only the stores wait for them
  ce = launch_k(tree_attn_tc_kernel, grid, dim3(AT_THREADS), smem, st, true, mkc, mvc, mkt, mvt, a);
  if (ce != cudaSuccess || a.NS == 1) return (int)ce;
  return launch_attn_combine(p, a.part_o, a.part_ml, a.NS, out, st);
}

}  // namespace medusa
