// Verification projection on the 5th-generation tensor cores ("Medusa Heads",
// "Attenzione sull'albero e accettazione": the base model scores every tree
// node; greedy acceptance needs its top choice, typical acceptance the
// entropy of its distribution).
//
//   logits[n][v] = o[n] . lm_head[v]   for every node n < N = B*T, token v < V,
//   reduced over v on the fly: argmax (ties to the lower id), max, and with a
//   temperature the softmax log-partition and entropy.  Logits never reach
//   global memory.
//
// Mapping (swap-AB): a tile is 256 vocabulary rows of lm_head, as two MMA
// M = 128 halves (A, K-major) that share every stage of the node operand (MMA
// N = BN <= 256 attention-output rows, K-major) -- the node operand is
// re-read from L2 once per tile, so a taller tile halves that traffic; K = H
// in blocks of 64 (one 128-byte swizzled TMA box per operand and stage).  The
// two accumulators fill the 512 TMEM columns.  Warp roles in a persistent CTA
// (one per SM):
//   warp 0      TMA producer (one thread), S-stage smem ring
//   warp 1      TMEM allocator + MMA issuer (one thread)
//   warps 2..    epilogue (four or two per TMEM lane quadrant by mode,
//               columns split in groups of 64): tcgen05.ld 16 columns at a time; per column
//               the max over the warp's rows and the lowest row reaching it
//               by a "transpose-reduce" across the lanes (each exchange
//               round halves the columns a lane carries: 15 pair exchanges
//               per 16 columns instead of 5 dependent rounds per column);
//               typical acceptance adds one exponential per element against
//               that max and the same reduction of (sum e, sum e*t).  The warps
//               combine in shared memory and write one partial (max, sum e,
//               sum e*t, argmax) per (vocab tile, node).
// A second small kernel merges the vocab-tile partials, one warp per node;
// with typical acceptance the same warp scores each child token of its node
// under the node's distribution (one dot product lm_head[token] . o_node)
// and writes the child's keep flag.
// Every wait is bounded; on a timeout the kernel sets MEDUSA_ERR_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and returns.
#include <limits.h>

#include "internal.cuh"
#include "tc.cuh"

namespace medusa {

constexpr int VT_M = 128;       // vocab rows per MMA (M)
constexpr int VT_SUB = 2;       // MMA halves per tile: a tile is VT_SUB * VT_M vocab rows
constexpr int VT_BK = 64;       // K elements per stage (128 bytes of bf16)
// Epilogue warps per mode: 16 for greedy and typical (four per TMEM lane
// quadrant, each a quarter of the columns: 33B step 4547 -> 4426 us; with the
// transpose-reduce epilogue the GQA-shaped typical step 614 -> 599 us), 8 for
// the sampling epilogues (two per quadrant: with 16 they spill registers).
__host__ __device__ constexpr int vt_epi_warps(int mode) { return mode <= 1 ? 16 : 8; }
__host__ __device__ constexpr int vt_threads(int mode) { return 64 + 32 * vt_epi_warps(mode); }
constexpr uint32_t VT_TMEM_COLS = 512;
constexpr uint64_t VT_WAIT_NS = 20ull * 1000 * 1000;  // 20 ms per wait

struct VtcArgs {
  int V, N, H, BN, n_vt, n_nt, n_tiles, nk, stages;  // V: lm_head rows this call holds
  int id_off;  // token id of lm_head row 0 (a vocabulary shard's first row)
  // overlap schedule of the fused step: the node operand is complete once
  // *node_ready reaches node_target (the tree attention's CTAs count
  // themselves); the producer waits for that instead of the preceding grid,
  // which cannot complete before the head projection it runs beside
  const int* node_ready;
  int node_target;
  uint32_t idesc;
  int typical;
  int sample;  // node choice = argmax of s / temperature + Gumbel noise
  uint32_t seed0, seed1;
  int step;
  float inv_temp;
  float4* part;  // [n_vt][N]: (max, sum e, sum e*t, argmax bits)
  int32_t* node_argmax;
  float* node_maxlogit;
  float* node_lse;
  float* node_entropy;
  uint8_t* ws;
  // typical acceptance: every child c of node n is scored under n's
  // distribution in the merge (keep[c] = p_n(token_c) > threshold_n)
  TreeDims td;
  int T;
  const int32_t* token;             // [B][T]
  const __nv_bfloat16* attn_out;    // [N][H]
  const __nv_bfloat16* lm_head;     // [V][H]
  uint8_t* keep;                    // [B][T]
  float log_eps, log_delta;
  float4* shard_out;  // a vocabulary shard: the merged state per node (max, sum e, sum e*t, argmax bits)
  // typical acceptance with a sampled bonus (MODE 3): per (vocab tile, node)
  // the best perturbed score s / temperature + g and its id, merged into
  // draw[node]
  float2* draw_part;  // [n_vt][N]
  int32_t* draw;      // [N]
};

struct Soft {
  float m, z, s;
  int i;
};

__device__ __forceinline__ Soft soft_empty() {
  Soft r;
  r.m = -INFINITY;
  r.z = 0.f;
  r.s = 0.f;
  r.i = INT_MAX;
  return r;
}

// merge of two column states; z == 0 is empty
__device__ __forceinline__ Soft soft_join(const Soft& a, const Soft& b, bool typical, float it) {
  if (a.z == 0.f) return b;
  if (b.z == 0.f) return a;
  Soft r;
  const bool af = better(a.m, a.i, b.m, b.i);
  r.m = af ? a.m : b.m;
  r.i = af ? a.i : b.i;
  if (typical) {
    const float da = (a.m - r.m) * it, db = (b.m - r.m) * it;
    const float ea = expf(da), eb = expf(db);
    r.z = a.z * ea + b.z * eb;
    r.s = ea * (a.s + a.z * da) + eb * (b.s + b.z * db);
  } else {
    r.z = a.z + b.z;
    r.s = 0.f;
  }
  return r;
}

// Best (value, id) of 16 columns over the warp's 32 lanes, each lane starting
// from its own best of the column: four exchange rounds that each hand half
// of the carried columns to the partner lane (8 + 4 + 2 + 1 pairs sent
// instead of 5 dependent rounds per column), then one round within the lane
// pair.  Lane l ends with column l >> 1 in bv[0], bi[0] (lanes l and l ^ 1
// agree).  Ties go to the lower id, so the result does not depend on the
// order of the merges.
__device__ __forceinline__ void best_transpose16(float (&bv)[16], int (&bi)[16], int lane) {
#pragma unroll
  for (int step = 0; step < 4; ++step) {
    const int o = 16 >> step, hh = 8 >> step;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < hh; ++k) {
      const float sv = up ? bv[k] : bv[k + hh], kv = up ? bv[k + hh] : bv[k];
      const int si = up ? bi[k] : bi[k + hh], ki = up ? bi[k + hh] : bi[k];
      const float rv = __shfl_xor_sync(0xffffffffu, sv, o);
      const int ri = __shfl_xor_sync(0xffffffffu, si, o);
      const bool take = better(rv, ri, kv, ki);
      bv[k] = take ? rv : kv;
      bi[k] = take ? ri : ki;
    }
  }
  const float rv = __shfl_xor_sync(0xffffffffu, bv[0], 1);
  const int ri = __shfl_xor_sync(0xffffffffu, bi[0], 1);
  if (better(rv, ri, bv[0], bi[0])) {
    bv[0] = rv;
    bi[0] = ri;
  }
}

__device__ __forceinline__ Soft shfl_soft(const Soft& a, int o) {
  Soft r;
  r.m = __shfl_xor_sync(0xffffffffu, a.m, o);
  r.z = __shfl_xor_sync(0xffffffffu, a.z, o);
  r.s = __shfl_xor_sync(0xffffffffu, a.s, o);
  r.i = __shfl_xor_sync(0xffffffffu, a.i, o);
  return r;
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds, each two 32x32->64-bit products of
// counter words with fixed multipliers, the high halves xored with the other
// words and the key; the key advances by a Weyl sequence between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// standard Gumbel noise -ln(-ln u) from the top 24 bits of a word (u strictly
// inside (0, 1), exact in fp32)
__device__ __forceinline__ float gumbel24(uint32_t x) {
  const float u = ((float)(x >> 8) + 0.5f) * (1.f / 16777216.f);
  return -__logf(-__logf(u));  // fast logarithm: the draws near a tie may differ from exact ones
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              uint8_t* ws) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::globaltimer_ns();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (tc::globaltimer_ns() - t0 > VT_WAIT_NS) {
      set_error(ws, MEDUSA_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// MODE: 0 greedy, 1 typical, 2 sample, 3 typical with a sampled bonus (a
// compile-time choice, so each instance carries only its own epilogue)
template <int MODE>
__global__ void __launch_bounds__(vt_threads(MODE), 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ VtcArgs a) {
  extern __shared__ uint8_t vt_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(vt_smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  const uint32_t bytesA1 = VT_M * VT_BK * 2, bytesA = VT_SUB * bytesA1, bytesB = (uint32_t)a.BN * VT_BK * 2;
  const uint32_t stage_bytes = bytesA + bytesB;
  Soft* red = reinterpret_cast<Soft*>(smem + (size_t)S * stage_bytes);  // [4][BN]
  float2* red2 = reinterpret_cast<float2*>(red + 4 * a.BN);               // MODE 3: [4][BN] draws
  uint64_t* bars = reinterpret_cast<uint64_t*>(red2 + (MODE == 3 ? 4 * a.BN : 0));
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* ep_ok = reinterpret_cast<volatile int*>(tmem_slot + 3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool typical = MODE == 1 || MODE == 3;
  constexpr int VT_EPI_WARPS = vt_epi_warps(MODE);
  constexpr int VT_EPI_GROUPS = VT_EPI_WARPS / 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(&tfull[0], 1);
    tc::mbar_init(&tempty[0], VT_EPI_WARPS);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, VT_TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      // lm_head is a weight no kernel writes: the first ring of its tiles is
      // requested before waiting for the kernel that produces the node operand
      const int first_t = blockIdx.x;
      const int npre = first_t < a.n_tiles ? (a.nk < S ? a.nk : S) : 0;
      for (int kb = 0; kb < npre; ++kb) {
        const int vt = first_t / a.n_nt;
        uint8_t* sa = smem + (size_t)kb * stage_bytes;
        tc::mbar_arrive_expect_tx(&full[kb], stage_bytes);
#pragma unroll
        for (int h = 0; h < VT_SUB; ++h)
          tc::tma_load_2d(sa + h * bytesA1, &tmA, &full[kb], kb * VT_BK, (vt * VT_SUB + h) * VT_M);
      }
      if (a.node_ready) {  // the node operand: every attention CTA has counted itself
        wait_count(a.node_ready, a.node_target, VT_WAIT_NS, a.ws);
        fence_proxy_async_global();
      } else {
        pdl_wait();  // the node operand is the previous kernel's output
      }
      for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x) {
        const int vt = t / a.n_nt, nt = t - vt * a.n_nt;
        for (int kb = 0; kb < a.nk; ++kb, ++g) {
          const int s = g % S;
          const uint32_t ph = (g / S) & 1u;
          uint8_t* sa = smem + (size_t)s * stage_bytes;
          if (g < (uint32_t)npre) {  // A already requested: add the node tile
            tc::tma_load_2d(sa + bytesA, &tmB, &full[s], kb * VT_BK, nt * a.BN);
            continue;
          }
          if (!wait_or_abort(&empty[s], ph ^ 1u, abort_flag, a.ws)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&full[s], stage_bytes);
#pragma unroll
          for (int h = 0; h < VT_SUB; ++h)
            tc::tma_load_2d(sa + h * bytesA1, &tmA, &full[s], kb * VT_BK, (vt * VT_SUB + h) * VT_M);
          tc::tma_load_2d(sa + bytesA, &tmB, &full[s], kb * VT_BK, nt * a.BN);
        }
      }
      if (!ok) {  // drain the copies this thread issued before leaving
        const uint32_t first = g > (uint32_t)S ? g - S : 0;
        for (uint32_t gi = first; gi < g; ++gi) {
          uint64_t* b = &full[gi % S];
          const uint64_t t0 = tc::globaltimer_ns();
          while (!tc::mbar_try_wait(b, (gi / S) & 1u) && tc::globaltimer_ns() - t0 < VT_WAIT_NS) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      uint32_t g = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x, ++tl) {
        const uint32_t aph = tl & 1u;  // one accumulator set (both halves), reused per tile
        if (!wait_or_abort(&tempty[0], aph ^ 1u, abort_flag, a.ws)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        for (int kb = 0; kb < a.nk; ++kb, ++g) {
          const int s = g % S;
          const uint32_t ph = (g / S) & 1u;
          if (!wait_or_abort(&full[s], ph, abort_flag, a.ws)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_u32(smem + (size_t)s * stage_bytes);
          const uint64_t db = tc::sw128_desc(sa + bytesA);
#pragma unroll
          for (int h = 0; h < VT_SUB; ++h) {
            const uint64_t da = tc::sw128_desc(sa + h * bytesA1);
#pragma unroll
            for (int j = 0; j < VT_BK / 16; ++j)  // K = 16 per MMA: +32 bytes in the swizzled row
              tc::mma_bf16(tmem + h * 256, da + 2 * j, db + 2 * j, a.idesc, (kb | j) != 0);
          }
          tc::mma_commit(&empty[s]);  // frees the stage once these MMAs have read it
        }
        if (!ok) break;
        tc::mma_commit(&tfull[0]);
      }
      // every MMA issued by this thread completes before TMEM is freed
      tc::mma_commit(drain);
      const uint64_t t0 = tc::globaltimer_ns();
      while (!tc::mbar_try_wait(drain, 0) && tc::globaltimer_ns() - t0 < VT_WAIT_NS) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    const int etid = threadIdx.x - 64;
    uint32_t tl = 0;
    for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++tl) {
      const int vt = t / a.n_nt, nt = t - vt * a.n_nt;
      const uint32_t aph = tl & 1u;
      // one thread waits, the named barrier hands its verdict to all 128
      if (etid == 0) *ep_ok = wait_or_abort(&tfull[0], aph, abort_flag, a.ws) ? 1 : 0;
      asm volatile("bar.sync 1, %0;" ::"r"(32 * VT_EPI_WARPS) : "memory");
      if (!*ep_ok) break;
      tc::fence_after_sync();
      // group g of the quadrant's warps (warps 2 + 4g .. 5 + 4g) takes every
      // VT_EPI_GROUPS-th group of 4 chunks of 16 columns, starting at group g
      const int grp = (warp - 2) >> 2;
      for (int ch0 = 4 * grp; ch0 < a.BN / 16; ch0 += 4 * VT_EPI_GROUPS) {
        const int nch = min(4, a.BN / 16 - ch0);
        if constexpr (typical) {
          // typical: per column the max and argmax as in greedy, then one
          // exponential per element against that max and a plain additive
          // transpose-reduce of (sum e, sum e*t) over the 64 rows
          const int row0 = vt * VT_SUB * VT_M + q * 32 + lane;  // half 1 adds VT_M
          const bool ok0 = row0 < a.V, ok1 = row0 + VT_M < a.V;
#pragma unroll 1
          for (int c = 0; c < nch; ++c) {
            float v[VT_SUB][16];
#pragma unroll
            for (int h = 0; h < VT_SUB; ++h)
              tc::tmem_ld16_nowait(tmem + h * 256 + ((uint32_t)(q * 32) << 16) + (ch0 + c) * 16, v[h]);
            tc::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < VT_SUB; ++h) tc::tmem_regs_ready(v[h]);
            // the column maxima and their rows first (transpose-reduce of
            // each lane's better row), then every lane fetches the 16 maxima
            float bv[16];
            int bi[16];
            float dv[16];  // MODE 3: the perturbed scores of the draw
            uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
            int di[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float x0 = ok0 ? v[0][j] : -INFINITY;
              const float x1 = ok1 ? v[1][j] : -INFINITY;
              const bool one = x1 > x0;  // equal values keep half 0 (the lower row)
              bv[j] = one ? x1 : x0;
              bi[j] = ok0 ? a.id_off + (one ? row0 + VT_M : row0) : INT_MAX;
              if constexpr (MODE == 3) {
                // the bonus draw: s / temperature + Gumbel noise, keyed as in the
                // sampling mode (one Philox call per row and 4 node columns)
                if ((j & 3) == 0) {
                  const uint32_t nc = (uint32_t)(nt * a.BN + (ch0 + c) * 16 + j) >> 2;
                  w0 = philox4x32_10(make_uint4((uint32_t)(a.id_off + row0), nc, (uint32_t)a.step, 0u), a.seed0,
                                     a.seed1);
                  w1 = philox4x32_10(make_uint4((uint32_t)(a.id_off + row0 + VT_M), nc, (uint32_t)a.step, 0u),
                                     a.seed0, a.seed1);
                }
                const uint32_t u0 = (j & 3) == 0 ? w0.x : (j & 3) == 1 ? w0.y : (j & 3) == 2 ? w0.z : w0.w;
                const uint32_t u1 = (j & 3) == 0 ? w1.x : (j & 3) == 1 ? w1.y : (j & 3) == 2 ? w1.z : w1.w;
                const float y0 = ok0 ? x0 * a.inv_temp + gumbel24(u0) : -INFINITY;
                const float y1 = ok1 ? x1 * a.inv_temp + gumbel24(u1) : -INFINITY;
                const bool one_d = y1 > y0;
                dv[j] = one_d ? y1 : y0;
                di[j] = ok0 ? a.id_off + (one_d ? row0 + VT_M : row0) : INT_MAX;
              }
            }
            best_transpose16(bv, bi, lane);
            if constexpr (MODE == 3) best_transpose16(dv, di, lane);
            const float colm = bv[0];  // column lane >> 1: max (-inf if no row is real) and its row
            const int coli = bi[0];
            float zs[16], ss[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float mj = __shfl_sync(0xffffffffu, colm, 2 * j);
              const bool any = mj > -INFINITY;
              const float x0 = ok0 ? v[0][j] : -INFINITY;
              const float x1 = ok1 ? v[1][j] : -INFINITY;
              const float t0 = ok0 && any ? (x0 - mj) * a.inv_temp : 0.f;
              const float t1 = ok1 && any ? (x1 - mj) * a.inv_temp : 0.f;
              // one hardware exp2 per element (exp2f), t stays in natural units for the sums
              const float e0 = ok0 && any ? exp2f(t0 * 1.4426950408889634f) : 0.f;
              const float e1 = ok1 && any ? exp2f(t1 * 1.4426950408889634f) : 0.f;
              zs[j] = e0 + e1;
              ss[j] = e0 * t0 + e1 * t1;
            }
            // after the four halving rounds lane l holds column l >> 1
#pragma unroll
            for (int step = 0; step < 4; ++step) {
              const int o = 16 >> step, hh = 8 >> step;
              const bool up = (lane & o) != 0;
#pragma unroll
              for (int k = 0; k < hh; ++k) {
                const float sz = up ? zs[k] : zs[k + hh], kz = up ? zs[k + hh] : zs[k];
                const float sv = up ? ss[k] : ss[k + hh], kv = up ? ss[k + hh] : ss[k];
                zs[k] = kz + __shfl_xor_sync(0xffffffffu, sz, o);
                ss[k] = kv + __shfl_xor_sync(0xffffffffu, sv, o);
              }
            }
            zs[0] += __shfl_xor_sync(0xffffffffu, zs[0], 1);
            ss[0] += __shfl_xor_sync(0xffffffffu, ss[0], 1);
            if ((lane & 1) == 0) {
              Soft o;
              o.m = colm;
              o.i = coli;
              o.z = coli == INT_MAX ? 0.f : zs[0];
              o.s = coli == INT_MAX ? 0.f : ss[0];
              red[q * a.BN + (ch0 + c) * 16 + (lane >> 1)] = o;
              if constexpr (MODE == 3) red2[q * a.BN + (ch0 + c) * 16 + (lane >> 1)] = make_float2(dv[0], __int_as_float(di[0]));
            }
          }
        } else {
          // greedy: per column, the best of this thread's two rows, then the
          // warp's best by a transpose-reduce (ties to the lowest row)
          const int row0 = vt * VT_SUB * VT_M + q * 32 + lane;  // half 1 adds VT_M
          const bool ok0 = row0 < a.V, ok1 = row0 + VT_M < a.V;
#pragma unroll
          for (int cp = 0; cp < 4; cp += 2) {  // two chunks (both halves) per TMEM wait
            if (cp >= nch) break;
            float v[VT_SUB][2][16];
#pragma unroll
            for (int h = 0; h < VT_SUB; ++h) {
              const uint32_t tb = tmem + h * 256 + ((uint32_t)(q * 32) << 16) + (ch0 + cp) * 16;
#pragma unroll
              for (int c = 0; c < 2; ++c)
                if (cp + c < nch) tc::tmem_ld16_nowait(tb + c * 16, v[h][c]);
            }
            tc::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < VT_SUB; ++h)
#pragma unroll
              for (int c = 0; c < 2; ++c) tc::tmem_regs_ready(v[h][c]);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              if (cp + c >= nch) break;
              Soft mine;
              mine.m = -INFINITY;
              mine.z = 0.f;
              mine.s = 0.f;
              mine.i = INT_MAX;
              if constexpr (MODE == 2) {  // s / temperature + Gumbel noise (one Philox call per 4 node columns)
                const uint32_t n0 = (uint32_t)(nt * a.BN + (ch0 + cp + c) * 16);
#pragma unroll
                for (int h = 0; h < VT_SUB; ++h) {
                  const uint32_t row = (uint32_t)(a.id_off + row0 + h * VT_M);  // the global token id
#pragma unroll
                  for (int j4 = 0; j4 < 16; j4 += 4) {
                    const uint4 w = philox4x32_10(make_uint4(row, (n0 + j4) >> 2, (uint32_t)a.step, 0u), a.seed0,
                                                  a.seed1);
                    v[h][c][j4] = v[h][c][j4] * a.inv_temp + gumbel24(w.x);
                    v[h][c][j4 + 1] = v[h][c][j4 + 1] * a.inv_temp + gumbel24(w.y);
                    v[h][c][j4 + 2] = v[h][c][j4 + 2] * a.inv_temp + gumbel24(w.z);
                    v[h][c][j4 + 3] = v[h][c][j4 + 3] * a.inv_temp + gumbel24(w.w);
                  }
                }
              }
              float bv[16];
              int bi[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float x0 = ok0 ? v[0][c][j] : -INFINITY;
                const float x1 = ok1 ? v[1][c][j] : -INFINITY;
                const bool one = x1 > x0;  // equal values keep half 0 (the lower row)
                bv[j] = one ? x1 : x0;
                bi[j] = ok0 ? a.id_off + (one ? row0 + VT_M : row0) : INT_MAX;
              }
              best_transpose16(bv, bi, lane);
              if (bi[0] != INT_MAX) {
                mine.m = bv[0];
                mine.i = bi[0];
                mine.z = 1.f;
              }
              if ((lane & 1) == 0) red[q * a.BN + (ch0 + cp + c) * 16 + (lane >> 1)] = mine;
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[0]);  // this warp is done with the accumulators
      asm volatile("bar.sync 1, %0;" ::"r"(32 * VT_EPI_WARPS) : "memory");
      for (int col = etid; col < a.BN; col += 32 * VT_EPI_WARPS) {
        const int n = nt * a.BN + col;
        if (n < a.N) {
          Soft m = red[col];
          for (int w = 1; w < 4; ++w) m = soft_join(m, red[w * a.BN + col], typical, a.inv_temp);
          a.part[(size_t)vt * a.N + n] = make_float4(m.m, m.z, m.s, __int_as_float(m.i));
          if constexpr (MODE == 3) {  // the draw: the larger perturbed score, ties to the lower id
            float2 d = red2[col];
            for (int w = 1; w < 4; ++w) {
              const float2 o = red2[w * a.BN + col];
              if (better(o.x, __float_as_int(o.y), d.x, __float_as_int(d.y))) d = o;
            }
            a.draw_part[(size_t)vt * a.N + n] = d;
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"r"(32 * VT_EPI_WARPS) : "memory");
    }
  }

  // ---------------------------------------------------------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, VT_TMEM_COLS);
  }
}

// Merges the per-tile partials of every node: one warp per node, each lane
// folds a strided subset of the vocab tiles (loads issued back to back), then
// a butterfly joins the 32 lane states.
template <bool TYPICAL>
__global__ void __launch_bounds__(256) verify_merge_kernel(const __grid_constant__ VtcArgs a) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_trigger();
  pdl_wait();
  if (n >= a.N) return;
  Soft m = soft_empty();
  for (int vt0 = 0; vt0 < a.n_vt; vt0 += 128) {
    float4 p[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int vt = vt0 + u * 32 + lane;
      p[u] = vt < a.n_vt ? a.part[(size_t)vt * a.N + n] : make_float4(-INFINITY, 0.f, 0.f, __int_as_float(INT_MAX));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      Soft o;
      o.m = p[u].x;
      o.z = p[u].y;
      o.s = p[u].z;
      o.i = __float_as_int(p[u].w);
      m = soft_join(m, o, TYPICAL, a.inv_temp);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = soft_join(m, shfl_soft(m, o), TYPICAL, a.inv_temp);
  if (a.shard_out) {  // the state itself: shards are combined after their exchange
    if (lane == 0) a.shard_out[n] = make_float4(m.m, m.z, m.s, __int_as_float(m.i));
    return;
  }
  if (TYPICAL && a.draw_part) {  // the bonus draw of this node: best perturbed score over the vocab tiles
    float dm = -INFINITY;
    int di = INT_MAX;
    for (int vt = lane; vt < a.n_vt; vt += 32) {
      const float2 d = a.draw_part[(size_t)vt * a.N + n];
      if (better(d.x, __float_as_int(d.y), dm, di)) {
        dm = d.x;
        di = __float_as_int(d.y);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, dm, o);
      const int oi = __shfl_xor_sync(0xffffffffu, di, o);
      if (better(om, oi, dm, di)) {
        dm = om;
        di = oi;
      }
    }
    if (lane == 0) a.draw[n] = di;
  }
  const float lz = logf(m.z);
  const float lse = m.m * a.inv_temp + lz, ent = lz - m.s / m.z;
  if (lane == 0) {
    a.node_argmax[n] = m.i;
    a.node_maxlogit[n] = m.m;
    if (TYPICAL) {
      a.node_lse[n] = lse;
      a.node_entropy[n] = ent;
    }
  }
  if (!TYPICAL) return;
  // children of this node (consecutive nodes): the child's token under this
  // node's softmax at the temperature, against the threshold
  const int b = n / a.T, i = n - b * a.T;
  const int kc = a.td.n_child[i];
  const int c0 = a.td.first_child[i];
  const float logthr = fminf(a.log_eps, a.log_delta - ent);
  const uint4* on = reinterpret_cast<const uint4*>(a.attn_out + (size_t)n * a.H);
  for (int r = 0; r < kc; ++r) {
    const int c = c0 + r;
    const int t = a.token[(size_t)b * a.T + c];
    const bool t_ok = t >= 0 && t < a.V;
    float s0 = 0.f, s1 = 0.f;
    if (t_ok) {
      const uint4* lr = reinterpret_cast<const uint4*>(a.lm_head + (size_t)t * a.H);
      for (int j = lane; j < a.H / 8; j += 32) {  // 8 bf16 per 16-byte load
        const uint4 x = __ldg(lr + j), y = __ldg(on + j);
        s0 = fmaf(bf16_lo(x.x), bf16_lo(y.x), s0);
        s1 = fmaf(bf16_hi(x.x), bf16_hi(y.x), s1);
        s0 = fmaf(bf16_lo(x.y), bf16_lo(y.y), s0);
        s1 = fmaf(bf16_hi(x.y), bf16_hi(y.y), s1);
        s0 = fmaf(bf16_lo(x.z), bf16_lo(y.z), s0);
        s1 = fmaf(bf16_hi(x.z), bf16_hi(y.z), s1);
        s0 = fmaf(bf16_lo(x.w), bf16_lo(y.w), s0);
        s1 = fmaf(bf16_hi(x.w), bf16_hi(y.w), s1);
      }
    }
    const float sdot = warp_sum(s0 + s1);
    if (lane == 0) {
      if (!t_ok) set_error(a.ws, MEDUSA_ERR_DEVICE);
      a.keep[(size_t)b * a.T + c] = t_ok && (sdot * a.inv_temp - lse > logthr);
    }
  }
}

// One CTA waits on an mbarrier that no thread or copy ever completes, with
// the same bounded wait as the kernels above, then reports the timeout.
__global__ void bounded_wait_probe_kernel(uint8_t* ws, uint64_t budget_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    if (!tc::mbar_wait(&bar, 0, budget_ns)) set_error(ws, MEDUSA_ERR_TIMEOUT);
  }
}

int launch_bounded_wait_probe(uint8_t* ws, uint64_t budget_ns, cudaStream_t st) {
  bounded_wait_probe_kernel<<<1, 32, 0, st>>>(ws, budget_ns);
  return (int)cudaGetLastError();
}

// ------------------------------------------------------------------- host --
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 [rows][cols] row-major, box of (64 columns x box_rows rows), 128-byte swizzle
int make_tmap_bf16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return (int)cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)VT_BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

// bf16 [depth][rows][cols] row-major, box of (64 columns x box_rows rows x 1),
// 128-byte swizzle; rows past `rows` (and columns past `cols`) read as zero
int make_tmap_bf16_3d(CUtensorMap* m, const void* base, int depth, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return (int)cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)depth};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
  cuuint32_t box[3] = {(cuuint32_t)VT_BK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

void verify_tc_shape(int N, int* BN, int* n_nt) {
  int nt = (N + 255) / 256;
  int bn = (N + nt - 1) / nt;
  bn = (bn + 15) / 16 * 16;
  if (bn < 16) bn = 16;
  *BN = bn;
  *n_nt = nt;
}

size_t verify_tc_part_bytes(int V, int N) {
  return (size_t)((V + VT_SUB * VT_M - 1) / (VT_SUB * VT_M)) * N * sizeof(float4);
}

int launch_verify_tc(const Plan& p, const void* attn_out, const void* lm_head, const int32_t* token, int32_t* node_argmax,
                     float* node_maxlogit, float* node_lse, float* node_entropy, uint8_t* ws, cudaStream_t st,
                     VerifyPart part, float4* shard_out) {
  VtcArgs a;
  a.V = p.Vs;
  a.id_off = p.v0;
  a.N = p.B * p.T;
  a.H = p.H;
  verify_tc_shape(a.N, &a.BN, &a.n_nt);
  a.n_vt = (p.Vs + VT_SUB * VT_M - 1) / (VT_SUB * VT_M);
  a.n_tiles = a.n_vt * a.n_nt;
  a.nk = p.H / VT_BK;
  a.idesc = tc::idesc_bf16_f32(VT_M, a.BN);
  a.typical = p.typical ? 1 : 0;
  a.sample = p.sample ? 1 : 0;
  a.seed0 = p.seed[0];
  a.seed1 = p.seed[1];
  a.step = p.step;
  a.inv_temp = (p.typical || p.sample) ? 1.f / p.temperature : 1.f;
  a.part = reinterpret_cast<float4*>(ws + p.off_vtc_part);
  a.node_ready = p.overlap ? reinterpret_cast<const int*>(ws) + TICKET_ATTN_DONE : nullptr;
  a.node_target = p.overlap ? (int)attn_tc_unsplit_ctas(p) : 0;
  a.node_argmax = node_argmax;
  a.node_maxlogit = node_maxlogit;
  a.node_lse = node_lse;
  a.node_entropy = node_entropy;
  a.ws = ws;
  a.td = p.tree;
  a.T = p.T;
  a.token = token;
  a.attn_out = reinterpret_cast<const __nv_bfloat16*>(attn_out);
  a.lm_head = reinterpret_cast<const __nv_bfloat16*>(lm_head);
  a.keep = ws + p.off_keep;
  a.shard_out = part == VERIFY_SHARD ? shard_out : nullptr;
  a.draw_part = p.sample_bonus ? reinterpret_cast<float2*>(ws + p.off_draw_part) : nullptr;
  a.draw = p.sample_bonus ? reinterpret_cast<int32_t*>(ws + p.off_draw) : nullptr;
  a.log_eps = p.typical ? logf(p.eps) : 0.f;
  a.log_delta = p.typical && p.delta > 0.f ? logf(p.delta) : -INFINITY;
  const unsigned mgrid = (unsigned)((a.N + 7) / 8);
  if (part == VERIFY_MERGE || part == VERIFY_SHARD) {
    if (a.typical) return (int)launch_k(verify_merge_kernel<true>, dim3(mgrid), dim3(256), 0, st, true, a);
    return (int)launch_k(verify_merge_kernel<false>, dim3(mgrid), dim3(256), 0, st, true, a);
  }
  const size_t stage = (size_t)(VT_SUB * VT_M + a.BN) * VT_BK * 2;
  const size_t fixed = 1024 + (size_t)4 * a.BN * (sizeof(Soft) + (p.sample_bonus ? sizeof(float2) : 0)) + 256;
  const size_t budget = 227 * 1024;
  int S = (int)((budget - fixed) / stage);
  if (S > 8) S = 8;
  if (S < 2) return (int)cudaErrorInvalidConfiguration;
  a.stages = S;
  const size_t smem = fixed + (size_t)S * stage;
  CUtensorMap tA, tB;
  int e = make_tmap_bf16(&tA, lm_head, p.Vs, p.H, VT_M);
  if (e) return e;
  e = make_tmap_bf16(&tB, attn_out, a.N, p.H, a.BN);
  if (e) return e;
  void (*kern)(CUtensorMap, CUtensorMap, VtcArgs) =
      p.sample_bonus ? verify_tc_kernel<3>
                     : (a.typical ? verify_tc_kernel<1> : (a.sample ? verify_tc_kernel<2> : verify_tc_kernel<0>));
  cudaError_t ce = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.n_tiles < p.sm_count ? a.n_tiles : p.sm_count;
  const int mode = p.sample_bonus ? 3 : (a.typical ? 1 : (a.sample ? 2 : 0));
  ce = launch_k(kern, dim3(grid), dim3(vt_threads(mode)), smem, st, true, tA, tB, a);
  if (ce != cudaSuccess || part == VERIFY_GEMM) return (int)ce;
  if (a.typical) return (int)launch_k(verify_merge_kernel<true>, dim3(mgrid), dim3(256), 0, st, true, a);
  return (int)launch_k(verify_merge_kernel<false>, dim3(mgrid), dim3(256), 0, st, true, a);
}

}  // namespace medusa
