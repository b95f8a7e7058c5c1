// Medusa heads on the 5th-generation tensor cores, bf16, batches 1..32
// ("Medusa Heads": head k maps the last
// hidden state h to z_k = h + SiLU(W1_k h + b1_k) and scores the vocabulary
// with W2_k z_k; the top-k tokens of every head build the candidate tree).
//
// Two launches of one kernel template:
//   layer       Z = W1_k . h for all sequences, epilogue adds b1, applies
//               SiLU and the residual, and stores z in bf16 as a hi/lo pair
//               (z_hi = bf16(z), z_lo = bf16(z - z_hi): rows 2b and 2b+1 of
//               the projection operand), so the bf16 projection keeps ~16
//               significant bits of z
//   projection  logits = W2_k . [z_hi; z_lo], epilogue sums the pair per
//               sequence and keeps each CTA's per-head top-k candidates
//               (merged per head by the tree kernel that follows).
//
// Mapping (swap-AB): weight rows are the MMA M dimension (tiles of 128 rows
// of one head, K-major, read by 3-D TMA boxes with the 128-byte swizzle, so a
// head's ragged last tile reads zeros), the sequences are N (<= 64).  A work
// unit is one tile x 128 reduction elements (two 64-wide boxes); each CTA
// takes a contiguous run of units (stream-K), so every CTA streams the same
// number of weight bytes; the grid is capped at 5/6 of the SMs (measured
// faster than all of them; the rest host the attention's early CTAs).  A
// tile cut by a CTA boundary is finished by
// whichever of its two CTAs arrives second at a per-boundary ticket: both
// store their partial accumulators, the second adds the other's and runs the
// epilogue (no CTA ever waits for another).  Warp roles per CTA (one CTA per
// SM): warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer, warps 2..5
// epilogue (one per TMEM lane quadrant), two accumulator buffers so the
// epilogue of one tile overlaps the MMAs of the next.  Every wait is bounded.
#include <limits.h>

#include "internal.cuh"
#include "tc.cuh"

namespace medusa {

int make_tmap_bf16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows);
int make_tmap_bf16_3d(CUtensorMap* m, const void* base, int depth, int rows, int cols, int box_rows);

constexpr int HT_M = 128;        // weight rows per tile (MMA M)
constexpr int HT_BK = 64;        // reduction elements per TMA box (128 bytes)
constexpr int HT_KB = 2;         // boxes per stage: a unit reduces 128 elements
constexpr int HT_EPI_WARPS = 4;  // one per TMEM lane quadrant
constexpr int HT_THREADS = 64 + 32 * HT_EPI_WARPS;
constexpr uint64_t HT_WAIT_NS = 20ull * 1000 * 1000;  // 20 ms per wait

struct HtArgs {
  int rows;      // rows per head: H for the layer, V for the projection
  int H;         // reduction length
  int K, B;      // heads, sequences
  int tps, nks;  // tiles per head, units per tile
  int U, upc;    // units in total, units per CTA
  int stages;
  uint32_t idesc;
  // layer
  const __nv_bfloat16* h;   // [B][H]
  const __nv_bfloat16* b1;  // [K][H]
  __nv_bfloat16* zs;        // [K][NZ][H]: row 2b = z_hi of sequence b, 2b+1 = z_lo
  int NZ;
  // projection
  int id_off;  // token id of local row 0 (a vocabulary shard's first row)
  int kmax;
  int topk_n[MEDUSA_MAX_HEADS];
  float* cand_val;  // [grid][kMaxPieces][B][kmax]
  int* cand_idx;
  int* cand_seg;    // [grid][kMaxPieces]
  // tiles cut by a CTA boundary
  float* slot;    // [kHeadsTcMaxCtas][2][N][128] partial accumulators
  int* tk_own;    // [kHeadsTcMaxCtas] this kernel's boundary tickets
  int* tk_other;  // the other heads kernel's tickets, cleared here
  // in medusa_step the projection lets the kernels after it start only once
  // its own wait has returned (so they start after the step's earlier work is
  // complete), and each of its CTAs counts itself into *proj_done when its
  // last output is written (the candidate merge waits for that count instead
  // of its preceding grid); the layer clears the count
  int late_trigger;
  int* proj_done;
  int* attn_done;  // layer: the tree attention's completion count, cleared with proj_done
  uint8_t* ws;
};

__device__ __forceinline__ bool ht_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint8_t* ws) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::globaltimer_ns();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (tc::globaltimer_ns() - t0 > HT_WAIT_NS) {
      set_error(ws, MEDUSA_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// A top-kn list in KM registers, best first, kept in the LAST kn slots: the
// first KM - kn slots hold sentinels that beat every value and are never
// displaced, so the admission threshold is always the last slot (a static
// register; a select on kn would be turned into a local-memory index).
template <int KM>
__device__ __forceinline__ void ht_reset(float (&lv)[KM], int (&li)[KM], int kn) {
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    const bool sentinel = j < KM - kn;
    lv[j] = sentinel ? INFINITY : -INFINITY;
    li[j] = sentinel ? -1 : INT_MAX;
  }
}

// sorted insertion (compare-and-swap chain; the sentinels never move)
template <int KM>
__device__ __forceinline__ void ht_insert(float (&lv)[KM], int (&li)[KM], float v, int id) {
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    const bool sw = better(v, id, lv[j], li[j]);
    const float ov = lv[j];
    const int oi = li[j];
    lv[j] = sw ? v : ov;
    li[j] = sw ? id : oi;
    v = sw ? ov : v;
    id = sw ? oi : id;
  }
}

__device__ __forceinline__ int ht_kept(const HtArgs& a, int seg) {
  int kn = 1;
#pragma unroll
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k)
    if (k == seg) kn = a.topk_n[k];
  return kn;
}

// End of a head's run in this CTA: the four epilogue warps' lists of each
// sequence are merged by the first epilogue warp (lane b takes sequence b)
// into the CTA's candidate slot `piece`.
template <int KM>
__device__ __forceinline__ void ht_flush(const HtArgs& a, const float (&lv)[KM], const int (&li)[KM], float* xv,
                                         int* xi, int cur_seg, int& piece, int q, int warp, int lane) {
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    xv[(q * 32 + lane) * KM + j] = lv[j];
    xi[(q * 32 + lane) * KM + j] = li[j];
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  const int kn = ht_kept(a, cur_seg);
  if (warp == 2 && lane < a.B) {
    float mv[KM];
    int mi[KM];
    ht_reset<KM>(mv, mi, kn);
    for (int w = 0; w < HT_EPI_WARPS; ++w)
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        const int id = xi[(w * 32 + lane) * KM + j];
        if (id >= 0) ht_insert<KM>(mv, mi, xv[(w * 32 + lane) * KM + j], id);
      }
    const size_t base = ((size_t)(blockIdx.x * kMaxPieces + piece) * a.B + lane) * a.kmax;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      const int r = j - (KM - kn);  // rank of slot j
      if (r >= 0 && r < a.kmax) {
        a.cand_val[base + r] = mv[j];
        a.cand_idx[base + r] = mi[j];
      }
    }
    for (int r = kn; r < a.kmax; ++r) {
      a.cand_val[base + r] = -INFINITY;
      a.cand_idx[base + r] = INT_MAX;
    }
  }
  if (warp == 2 && lane == 0) a.cand_seg[blockIdx.x * kMaxPieces + piece] = cur_seg;
  asm volatile("bar.sync 1, 128;" ::: "memory");
  ++piece;
}

template <int EPI, int N, int KM>
__global__ void __launch_bounds__(HT_THREADS, 1)
    heads_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, HtArgs a) {
  extern __shared__ uint8_t ht_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ht_smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t bytesA1 = HT_M * HT_BK * 2, bytesB1 = N * HT_BK * 2;
  constexpr uint32_t stage_bytes = HT_KB * (bytesA1 + bytesB1);
  constexpr uint32_t tmem_cols = 2 * N < 32 ? 32 : 2 * N;
  const int S = a.stages;
  float* xv = reinterpret_cast<float*>(smem + (size_t)S * stage_bytes);  // [4][32][KM] list exchange
  int* xi = reinterpret_cast<int*>(xv + HT_EPI_WARPS * 32 * KM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(xi + HT_EPI_WARPS * 32 * KM);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* ep_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u0 = blockIdx.x * a.upc;
  const int u1 = min(a.U, u0 + a.upc);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], HT_EPI_WARPS);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (!a.late_trigger) pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane != 0 && a.late_trigger) {
      pdl_wait();
      pdl_trigger();
    }
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      auto load_a = [&](uint8_t* sa, uint64_t* bar, int u) {
        const int t = u / a.nks, ks = u - t * a.nks, seg = t / a.tps, tt = t - seg * a.tps;
#pragma unroll
        for (int j = 0; j < HT_KB; ++j)
          tc::tma_load_3d(sa + j * bytesA1, &tmA, bar, (ks * HT_KB + j) * HT_BK, tt * HT_M, seg);
      };
      auto load_b = [&](uint8_t* sb, uint64_t* bar, int u) {
        const int t = u / a.nks, ks = u - t * a.nks, seg = t / a.tps;
#pragma unroll
        for (int j = 0; j < HT_KB; ++j)
          tc::tma_load_2d(sb + j * bytesB1, &tmB, bar, (ks * HT_KB + j) * HT_BK, EPI == 0 ? 0 : seg * N);
      };
      // the weights are written by no kernel: the first ring of weight boxes
      // is requested before waiting for the kernel that produces the operand
      const int npre = min(u1 - u0, S);
      for (int i = 0; i < npre; ++i) {
        uint8_t* sa = smem + (size_t)i * stage_bytes;
        tc::mbar_arrive_expect_tx(&full[i], stage_bytes);
        load_a(sa, &full[i], u0 + i);
      }
      pdl_wait();
      if (a.late_trigger) pdl_trigger();
      for (int u = u0; u < u1; ++u, ++g) {
        const int s = g % S;
        const uint32_t ph = (g / S) & 1u;
        uint8_t* sa = smem + (size_t)s * stage_bytes;
        if (g < (uint32_t)npre) {
          load_b(sa + HT_KB * bytesA1, &full[s], u);
          continue;
        }
        if (!ht_wait(&empty[s], ph ^ 1u, abort_flag, a.ws)) {
          ok = false;
          break;
        }
        tc::mbar_arrive_expect_tx(&full[s], stage_bytes);
        load_a(sa, &full[s], u);
        load_b(sa + HT_KB * bytesA1, &full[s], u);
      }
      if (!ok) {  // drain the copies this thread issued before leaving
        const uint32_t first = g > (uint32_t)S ? g - S : 0;
        for (uint32_t gi = first; gi < g; ++gi) {
          uint64_t* b = &full[gi % S];
          const uint64_t t0 = tc::globaltimer_ns();
          while (!tc::mbar_try_wait(b, (gi / S) & 1u) && tc::globaltimer_ns() - t0 < HT_WAIT_NS) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (a.late_trigger) {
      pdl_wait();
      pdl_trigger();
    }
    if (lane == 0) {
      uint32_t g = 0, tl = 0;
      bool ok = true;
      for (int u = u0; u < u1 && ok; ++tl) {
        const int t = u / a.nks;
        const int u_end = min(u1, (t + 1) * a.nks);
        const uint32_t buf = tl & 1u;
        if (!ht_wait(&tempty[buf], ((tl >> 1) & 1u) ^ 1u, abort_flag, a.ws)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        for (int uu = u; uu < u_end; ++uu, ++g) {
          const int s = g % S;
          if (!ht_wait(&full[s], (g / S) & 1u, abort_flag, a.ws)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_u32(smem + (size_t)s * stage_bytes);
#pragma unroll
          for (int j = 0; j < HT_KB; ++j) {
            const uint64_t da = tc::sw128_desc(sa + j * bytesA1);
            const uint64_t db = tc::sw128_desc(sa + HT_KB * bytesA1 + j * bytesB1);
#pragma unroll
            for (int kk = 0; kk < HT_BK / 16; ++kk)  // K = 16 per MMA: +32 bytes in the swizzled row
              tc::mma_bf16(tmem + buf * N, da + 2 * kk, db + 2 * kk, a.idesc, (uu != u || j != 0 || kk != 0));
          }
          tc::mma_commit(&empty[s]);
        }
        if (!ok) break;
        tc::mma_commit(&tfull[buf]);
        u = u_end;
      }
      tc::mma_commit(drain);  // every MMA of this thread completes before TMEM is freed
      const uint64_t t0 = tc::globaltimer_ns();
      while (!tc::mbar_try_wait(drain, 0) && tc::globaltimer_ns() - t0 < HT_WAIT_NS) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    const int etid = threadIdx.x - 64;
    pdl_wait();
    if (a.late_trigger) pdl_trigger();
    // the other heads kernel has completed (or not started, for the layer):
    // its tickets are reset for its next launch
    for (int i = blockIdx.x * (32 * HT_EPI_WARPS) + etid; i < kHeadsTcMaxCtas; i += gridDim.x * 32 * HT_EPI_WARPS)
      a.tk_other[i] = 0;
    if (EPI == 0 && blockIdx.x == 0 && etid == 0) {  // the previous step has completed
      *a.proj_done = 0;
      *a.attn_done = 0;
    }
    float lv[KM];
    int li[KM];
    ht_reset<KM>(lv, li, KM);
    int cur_seg = -1, piece = 0;
    uint32_t tl = 0;
    bool alive = u0 < u1;
    const int t_first = u0 / a.nks, t_last = alive ? (u1 - 1) / a.nks : -1;
    for (int t = t_first; t <= t_last; ++t, ++tl) {
      const uint32_t buf = tl & 1u;
      if (etid == 0) *ep_flag = ht_wait(&tfull[buf], (tl >> 1) & 1u, abort_flag, a.ws) ? 1 : 0;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (!*ep_flag) {
        alive = false;
        break;
      }
      tc::fence_after_sync();
      float acc[N];
      {
        float v[N / 16][16];
        const uint32_t tb = tmem + buf * N + ((uint32_t)(q * 32) << 16);
#pragma unroll
        for (int c = 0; c < N / 16; ++c) tc::tmem_ld16_nowait(tb + c * 16, v[c]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < N / 16; ++c) {
          tc::tmem_regs_ready(v[c]);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[c * 16 + j] = v[c][j];
        }
      }
      // the accumulators are in registers: the buffer may take the next tile
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[buf]);

      const bool cut_lo = (t == t_first) && (u0 % a.nks != 0);  // began in the previous CTA
      const bool cut_hi = (t == t_last) && (u1 % a.nks != 0);   // ends in the next CTA
      if (cut_lo || cut_hi) {
        const int boundary = cut_lo ? blockIdx.x - 1 : blockIdx.x;
        const int side = cut_lo ? 1 : 0;
        float* mine = a.slot + ((size_t)boundary * 2 + side) * N * HT_M + q * 32 + lane;
#pragma unroll
        for (int n = 0; n < N; ++n) mine[(size_t)n * HT_M] = acc[n];
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (etid == 0) *ep_flag = atomicAdd(&a.tk_own[boundary], 1);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (*ep_flag == 0) continue;  // the other CTA finishes this tile
        __threadfence();
        const float* other = a.slot + ((size_t)boundary * 2 + (1 - side)) * N * HT_M + q * 32 + lane;
#pragma unroll
        for (int n = 0; n < N; ++n) acc[n] += __ldcg(other + (size_t)n * HT_M);
      }

      const int seg = t / a.tps;
      const int row0 = (t - seg * a.tps) * HT_M + q * 32;  // row of lane 0 within the head
      const int row = row0 + lane;
      const bool valid = row < a.rows;
      if (EPI == 0) {
        // z = h + SiLU(W1 h + b1), stored as the bf16 pair (hi, lo)
        if (valid) {
          const float bias = __bfloat162float(a.b1[(size_t)seg * a.H + row]);
          __nv_bfloat16* zrow = a.zs + (size_t)seg * a.NZ * a.H + row;
#pragma unroll
          for (int b = 0; b < N; ++b) {
            if (b >= a.B) break;
            const float pre = acc[b] + bias;
            const float silu = pre / (1.f + expf(-pre));
            const float z = __bfloat162float(a.h[(size_t)b * a.H + row]) + silu;
            const __nv_bfloat16 hi = __float2bfloat16_rn(z);
            const __nv_bfloat16 lo = __float2bfloat16_rn(z - __bfloat162float(hi));
            zrow[(size_t)(2 * b) * a.H] = hi;
            zrow[(size_t)(2 * b + 1) * a.H] = lo;
          }
        }
      } else {
        if (seg != cur_seg) {
          if (cur_seg >= 0) ht_flush<KM>(a, lv, li, xv, xi, cur_seg, piece, q, warp, lane);
          cur_seg = seg;
          ht_reset<KM>(lv, li, ht_kept(a, seg));
        }
        // per sequence b: the rows of this warp that beat the kn-th entry of
        // the warp's list (held by lane b) enter it, best first
#pragma unroll
        for (int b = 0; b < N / 2; ++b) {
          if (b >= a.B) break;
          const float v = valid ? acc[2 * b] + acc[2 * b + 1] : -INFINITY;
          const int r = valid ? a.id_off + row : INT_MAX;
          float tv = __shfl_sync(0xffffffffu, lv[KM - 1], b);
          int ti = __shfl_sync(0xffffffffu, li[KM - 1], b);
          unsigned pass = __ballot_sync(0xffffffffu, valid && better(v, r, tv, ti));
          while (pass) {
            const bool in = (pass >> lane) & 1u;
            const int key = in ? order_key(v) : INT_MIN;
            int kmx;
            asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(kmx) : "r"(key));
            const unsigned top = __ballot_sync(0xffffffffu, in && key == kmx);
            const int w = __ffs(top) - 1;  // lowest lane = lowest row among equal values
            const float wv = __shfl_sync(0xffffffffu, v, w);
            if (lane == b) ht_insert<KM>(lv, li, wv, a.id_off + row0 + w);
            pass &= ~(1u << w);
            tv = __shfl_sync(0xffffffffu, lv[KM - 1], b);
            ti = __shfl_sync(0xffffffffu, li[KM - 1], b);
            pass &= __ballot_sync(0xffffffffu, valid && better(v, r, tv, ti));
          }
        }
      }
    }
    if (EPI == 1 && alive) {
      if (cur_seg >= 0) ht_flush<KM>(a, lv, li, xv, xi, cur_seg, piece, q, warp, lane);
      if (warp == 2 && lane == 0)
        for (int p = piece; p < kMaxPieces; ++p) a.cand_seg[blockIdx.x * kMaxPieces + p] = -1;
    }
  }

  // ---------------------------------------------------------------- teardown
  if (EPI == 1 && a.proj_done) __threadfence();  // this thread's outputs, before the count below
  tc::fence_before_sync();
  __syncthreads();
  if (EPI == 1 && a.proj_done && threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.proj_done, 1);
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
}

// ------------------------------------------------------------------- host --
static int ht_n_layer(int B) { return B <= 16 ? 16 : 32; }
static int ht_n_proj(int B) { return 2 * B <= 16 ? 16 : (2 * B <= 32 ? 32 : 64); }

bool heads_tc_supported(const Plan& p) { return p.bf16 && p.B <= kHeadsTcMaxBatch; }

size_t heads_tc_zs_bytes(int K, int B, int H) { return (size_t)K * ht_n_proj(B) * H * 2; }
size_t heads_tc_slot_bytes(int B) {
  const int n = ht_n_proj(B) > ht_n_layer(B) ? ht_n_proj(B) : ht_n_layer(B);
  return (size_t)kHeadsTcMaxCtas * 2 * n * HT_M * sizeof(float);
}

// stream-K partition: units per CTA and grid
static void ht_partition(const Plan& p, int rows, HtArgs* a, int* grid) {
  a->nks = (p.H + HT_KB * HT_BK - 1) / (HT_KB * HT_BK);
  a->tps = (rows + HT_M - 1) / HT_M;
  a->U = p.K * a->tps * a->nks;
  const int cmax = p.heads_ctas < kHeadsTcMaxCtas ? p.heads_ctas : kHeadsTcMaxCtas;
  int upc = (a->U + cmax - 1) / cmax;
  if (upc < a->nks) upc = a->nks;  // a tile is cut at most once
  a->upc = upc;
  *grid = (a->U + upc - 1) / upc;
}

int heads_tc_proj_grid(const Plan& p) {
  HtArgs a{};
  int grid = 0;
  ht_partition(p, p.Vs, &a, &grid);
  return grid;
}

template <int EPI, int N, int KM>
static int ht_launch(const CUtensorMap& tA, const CUtensorMap& tB, HtArgs a, int grid, bool pdl, cudaStream_t st) {
  constexpr size_t stage = (size_t)HT_KB * (HT_M + N) * HT_BK * 2;
  const size_t fixed = 1024 + (size_t)HT_EPI_WARPS * 32 * KM * 8 + 512;
  int S = (int)((227 * 1024 - fixed) / stage);
  if (S > 8) S = 8;
  if (S < 2) return (int)cudaErrorInvalidConfiguration;
  a.stages = S;
  a.idesc = tc::idesc_bf16_f32(HT_M, N);
  const size_t smem = fixed + (size_t)S * stage;
  auto k = heads_tc_kernel<EPI, N, KM>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_k(k, dim3(grid), dim3(HT_THREADS), smem, st, pdl, tA, tB, a);
}

static void ht_common(const Plan& p, uint8_t* ws, HtArgs* a) {
  a->H = p.H;
  a->K = p.K;
  a->B = p.B;
  a->NZ = ht_n_proj(p.B);
  a->zs = reinterpret_cast<__nv_bfloat16*>(ws + p.off_zs);
  a->slot = reinterpret_cast<float*>(ws + p.off_ht_slot);
  a->ws = ws;
  a->late_trigger = 0;
  a->proj_done = nullptr;
}

int launch_fc_tc(const Plan& p, const void* h, const void* W1, const void* b1, uint8_t* ws, cudaStream_t st) {
  HtArgs a{};
  ht_common(p, ws, &a);
  a.rows = p.H;
  a.h = reinterpret_cast<const __nv_bfloat16*>(h);
  a.b1 = reinterpret_cast<const __nv_bfloat16*>(b1);
  a.tk_own = reinterpret_cast<int*>(ws + p.off_ht_tickets);
  a.tk_other = a.tk_own + kHeadsTcMaxCtas;
  a.proj_done = reinterpret_cast<int*>(ws) + TICKET_PROJ_DONE;
  a.attn_done = reinterpret_cast<int*>(ws) + TICKET_ATTN_DONE;
  int grid = 0;
  ht_partition(p, p.H, &a, &grid);
  if (a.upc > a.tps * a.nks) return (int)cudaErrorInvalidConfiguration;  // a CTA must touch at most 2 heads
  const int n = ht_n_layer(p.B);
  CUtensorMap tA, tB;
  int e = make_tmap_bf16_3d(&tA, W1, p.K, p.H, p.H, HT_M);
  if (e) return e;
  e = make_tmap_bf16(&tB, h, p.B, p.H, n);
  if (e) return e;
  // programmatic dependent launch: W1 boxes stream before the wait, h and the
  // outputs after it
  if (n == 16) return ht_launch<0, 16, 4>(tA, tB, a, grid, true, st);
  return ht_launch<0, 32, 4>(tA, tB, a, grid, true, st);
}

int launch_proj_tc_only(const Plan& p, const void* W2, uint8_t* ws, cudaStream_t st, int* ctas, int* upc,
                        int* ups) {
  HtArgs a{};
  ht_common(p, ws, &a);
  a.rows = p.Vs;
  a.id_off = p.v0;
  a.kmax = p.kmax;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.topk_n[k] = p.topk_n[k];
  a.cand_val = reinterpret_cast<float*>(ws + p.off_cand_val);
  a.cand_idx = reinterpret_cast<int*>(ws + p.off_cand_idx);
  a.cand_seg = reinterpret_cast<int*>(ws + p.off_cand_seg);
  a.tk_other = reinterpret_cast<int*>(ws + p.off_ht_tickets);
  a.tk_own = a.tk_other + kHeadsTcMaxCtas;
  if (p.overlap || p.late_tree) {  // see HtArgs: dependents start after the wait, CTAs count themselves
    a.late_trigger = 1;
    a.proj_done = reinterpret_cast<int*>(ws) + TICKET_PROJ_DONE;
  }
  int grid = 0;
  ht_partition(p, p.Vs, &a, &grid);
  if (a.upc > a.tps * a.nks) return (int)cudaErrorInvalidConfiguration;  // a CTA must touch at most 2 heads
  *ctas = grid;
  *upc = a.upc;
  *ups = a.tps * a.nks;
  const int n = ht_n_proj(p.B);
  CUtensorMap tA, tB;
  int e = make_tmap_bf16_3d(&tA, W2, p.K, p.Vs, p.H, HT_M);
  if (e) return e;
  e = make_tmap_bf16(&tB, a.zs, p.K * n, p.H, n);
  if (e) return e;
#define HT_PICK(NN)                                                              \
  if (n == NN) {                                                                 \
    if (p.kmax <= 4) return ht_launch<1, NN, 4>(tA, tB, a, grid, true, st);      \
    if (p.kmax <= 8) return ht_launch<1, NN, 8>(tA, tB, a, grid, true, st);      \
    return ht_launch<1, NN, MEDUSA_MAX_TOPK>(tA, tB, a, grid, true, st);         \
  }
  HT_PICK(16)
  HT_PICK(32)
  HT_PICK(64)
#undef HT_PICK
  return (int)cudaErrorInvalidValue;
}

int launch_topk_merge(const Plan& p, int32_t* topk_idx, float* topk_val, uint8_t* ws, int ctas, int rpc, int S,
                      cudaStream_t st);

int launch_proj_tc(const Plan& p, const void* W2, int32_t* topk_idx, float* topk_val, uint8_t* ws, cudaStream_t st) {
  int ctas = 0, upc = 0, ups = 0;
  int e = launch_proj_tc_only(p, W2, ws, st, &ctas, &upc, &ups);
  if (e) return e;
  return launch_topk_merge(p, topk_idx, topk_val, ws, ctas, upc, ups, st);
}

}  // namespace medusa
