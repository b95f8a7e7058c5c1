// Weight-streaming row kernel: out[c][r] = W[r] . x[c, seg(r)] for every row r
// of a [R][H] weight and every column c (a batch row or a tree node), with
// the reduction over rows fused into the epilogue:
//   EPI_FC     -- Medusa head layer: z[c][k][j] = h[c][j] + SiLU(acc + b1[k][j])
//                 (W1 rows, segment = head k)            ["Medusa Heads",
//                 "Come le teste prevedono i token successivi"]
//   EPI_TOPK   -- head vocabulary projection + per-head top-k of each column
//                 (W2 rows, segment = head k)            [same section, and
//                 "Attenzione sull'albero e accettazione": best tokens per head]
//   EPI_VERIFY -- base lm_head over tree nodes: argmax, max and (typical)
//                 softmax log-partition / entropy of each column
//                                                        ["Attenzione sull'albero
//                 e accettazione": the base model's choice at every node]
//
// Design (HBM-bound at small column counts): a persistent grid of
// sm_count * occupancy CTAs splits the R rows into equal contiguous ranges
// (balanced to one row); each warp streams whole rows with 16-byte
// L1-bypassing loads, 16 loads in flight per lane, against x held in shared
// memory as fp32; fp32 accumulation; one warp reduction per (row, column).
// Per-CTA partial results (top-k lists or softmax states) go to the
// workspace and the last CTA to finish (atomic ticket, no waiting) merges
// them, so one launch produces the final answer.
#include <float.h>
#include <limits.h>

#include "internal.cuh"

namespace medusa {

enum Epi { EPI_FC = 0, EPI_TOPK = 1, EPI_VERIFY = 2 };
constexpr int KMAX = MEDUSA_MAX_TOPK;  // compile-time bound of a top-k list
constexpr int UNROLL = 16;           // 16-byte loads in flight per lane
constexpr int kRowBuf = 2048;        // EPI_TOPK: rows a CTA may own (row results kept in shared memory)

struct RowArgs {
  const void* W;  // [R][H]
  const void* x;  // x(c, seg, j) = x[c * x_cs + seg * x_ss + j]
  long long x_cs, x_ss;
  int R, S, H, C, rpc, nseg;
  uint8_t* ws;
  int* ticket;
  // EPI_FC
  const void* bias;  // [nseg][H]
  float* z;          // [C][nseg][H]
  // EPI_TOPK
  int kmax;
  int topk_n[MEDUSA_MAX_HEADS];
  float* cand_val;  // [ctas][kMaxPieces][C][kmax]
  int* cand_idx;
  int* cand_seg;  // [ctas][kMaxPieces]
  int32_t* out_idx;
  float* out_val;  // [C][nseg][kmax]
  // EPI_VERIFY
  int typical;
  float inv_temp;
  float* part;    // [ctas][C][3] = (max, sum e, sum e*t), t = (x - max) * inv_temp
  int* part_idx;  // [ctas][C]
  int32_t* node_argmax;
  float* node_maxlogit;
  float* node_lse;
  float* node_entropy;
  float4* soft_out;  // a vocabulary shard: the merged state (max, sum e, sum e*t, argmax bits) per column instead
  int id_off;        // EPI_TOPK / EPI_VERIFY: token id of local row 0
};

// ---------------------------------------------------------------- helpers --
// topk_n[seg] without a dynamic index into the kernel parameter block (which
// would copy the whole block to local memory)
__device__ __forceinline__ int kept_of(const RowArgs& a, int seg) {
  int n = 1;
#pragma unroll
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k)
    if (k == seg) n = a.topk_n[k];
  return n;
}

// insert (v, id) into a best-first list of n live entries (n <= KM): one
// compare-and-swap pass, branch-free so the list stays in registers
template <int KM>
__device__ __forceinline__ void list_insert(float (&lv)[KM], int (&li)[KM], int n, float v, int id) {
  float tv = lv[0];
  int ti = li[0];
#pragma unroll
  for (int i = 1; i < KM; ++i)  // last live entry, selected without a dynamic index
    if (i == n - 1) {
      tv = lv[i];
      ti = li[i];
    }
  if (!better(v, id, tv, ti)) return;
#pragma unroll
  for (int i = 0; i < KM; ++i) {
    const bool sw = (i < n) && better(v, id, lv[i], li[i]);
    const float ov = lv[i];
    const int oi = li[i];
    lv[i] = sw ? v : ov;
    li[i] = sw ? id : oi;
    v = sw ? ov : v;
    id = sw ? oi : id;
  }
}

template <int KM>
__device__ __forceinline__ void list_reset(float (&lv)[KM], int (&li)[KM]) {
#pragma unroll
  for (int i = 0; i < KM; ++i) {
    lv[i] = -INFINITY;
    li[i] = INT_MAX;
  }
}

// Warp-wide top-n of the union of the lanes' best-first lists: n rounds of
// "the best list head wins, its owner pops".  Lane 0 writes n_out entries
// (ranks >= n, or missing ones, get -inf and pad_idx).
template <int KM>
__device__ __forceinline__ void warp_select(float (&lv)[KM], int (&li)[KM], int n, int n_out, float* out_val,
                                            int* out_idx, int pad_idx) {
  const int lane = threadIdx.x & 31;
  for (int rnk = 0; rnk < n_out; ++rnk) {
    float bv = lv[0];
    int bi = li[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi != INT_MAX && lv[0] == bv && li[0] == bi) {  // ids are unique: exactly one owner
#pragma unroll
      for (int i = 0; i < KM - 1; ++i) {
        lv[i] = lv[i + 1];
        li[i] = li[i + 1];
      }
      lv[KM - 1] = -INFINITY;
      li[KM - 1] = INT_MAX;
    }
    if (lane == 0) {
      const bool live = rnk < n && bi != INT_MAX;
      out_val[rnk] = live ? bv : -INFINITY;
      out_idx[rnk] = live ? bi : pad_idx;
    }
  }
}

// softmax state of a column: max m (index mi), z = sum e^{t}, s = sum e^{t} t,
// t = (x - m) * it.  z == 0 means empty.
struct SoftState {
  float m, z, s;
  int mi;
};

__device__ __forceinline__ void soft_push(SoftState& st, float x, int id, bool typical, float it) {
  if (st.z == 0.f) {
    st.m = x;
    st.mi = id;
    st.z = 1.f;
    st.s = 0.f;
    return;
  }
  if (better(x, id, st.m, st.mi)) {
    if (typical) {
      float d = (st.m - x) * it;  // <= 0
      float sc = expf(d);
      st.s = sc * (st.s + st.z * d);
      st.z = st.z * sc + 1.f;
    } else {
      st.z += 1.f;
    }
    st.m = x;
    st.mi = id;
  } else if (typical) {
    float t = (x - st.m) * it;
    float e = expf(t);
    st.z += e;
    st.s += e * t;
  } else {
    st.z += 1.f;
  }
}

__device__ __forceinline__ SoftState soft_merge(SoftState a, SoftState b, bool typical, float it) {
  if (a.z == 0.f) return b;
  if (b.z == 0.f) return a;
  SoftState r;
  bool a_first = better(a.m, a.mi, b.m, b.mi);
  r.m = a_first ? a.m : b.m;
  r.mi = a_first ? a.mi : b.mi;
  if (typical) {
    float da = (a.m - r.m) * it, db = (b.m - r.m) * it;
    float ea = expf(da), eb = expf(db);
    r.z = a.z * ea + b.z * eb;
    r.s = ea * (a.s + a.z * da) + eb * (b.s + b.z * db);
  } else {
    r.z = a.z + b.z;
    r.s = 0.f;
  }
  return r;
}

// ------------------------------------------------------------------ kernel --
template <typename TW, typename TX, int NC, int EPI>
__global__ void __launch_bounds__(kThreads, 2) stream_rows_kernel(RowArgs a) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);  // [NC][H]
  float* rowbuf = xs + NC * a.H;                  // EPI_TOPK: [NC][kRowBuf] row results of a piece
  __shared__ SoftState wsoft[kWarps][NC];
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, c0 = blockIdx.y * NC;
  const int r_begin = cta * a.rpc;
  const int r_end = min(a.R, r_begin + a.rpc);
  constexpr int EPV = 16 / sizeof(TW);  // weight elements per 16-byte vector
  const int nvec = a.H / EPV;
  const bool typical = a.typical != 0;

  pdl_trigger();
  pdl_wait();
  SoftState soft;
  soft.m = -INFINITY;
  soft.z = 0.f;
  soft.s = 0.f;
  soft.mi = INT_MAX;

  int piece = 0;
  for (int r0 = r_begin; r0 < r_end && piece < kMaxPieces; ++piece) {
    const int seg = r0 / a.S;
    const int r1 = min(r_end, (seg + 1) * a.S);
    // ---- x tile of this segment into shared memory (fp32, zero past C)
    __syncthreads();
    for (int e = threadIdx.x; e < NC * a.H; e += kThreads) {
      const int c = e / a.H, j = e - c * a.H;
      float v = 0.f;
      if (c0 + c < a.C)
        v = to_f32(reinterpret_cast<const TX*>(a.x)[(long long)(c0 + c) * a.x_cs + (long long)seg * a.x_ss + j]);
      xs[e] = v;
    }
    __syncthreads();

    const int kn = (EPI == EPI_TOPK) ? kept_of(a, seg) : 1;

    for (int r = r0 + warp; r < r1; r += kWarps) {
      const uint4* wrow = reinterpret_cast<const uint4*>(reinterpret_cast<const TW*>(a.W) + (size_t)r * a.H);
      float acc[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] = 0.f;
      for (int base = 0; base < nvec; base += 32 * UNROLL) {
        uint4 w[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
          const int v = base + u * 32 + lane;
          w[u] = v < nvec ? ldg_stream(wrow + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
          const int v = base + u * 32 + lane;
          if (v < nvec) {
            float wf[8];
            if (sizeof(TW) == 2) {
              wf[0] = bf16_lo(w[u].x); wf[1] = bf16_hi(w[u].x);
              wf[2] = bf16_lo(w[u].y); wf[3] = bf16_hi(w[u].y);
              wf[4] = bf16_lo(w[u].z); wf[5] = bf16_hi(w[u].z);
              wf[6] = bf16_lo(w[u].w); wf[7] = bf16_hi(w[u].w);
            } else {
              wf[0] = __uint_as_float(w[u].x); wf[1] = __uint_as_float(w[u].y);
              wf[2] = __uint_as_float(w[u].z); wf[3] = __uint_as_float(w[u].w);
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              const float4* xp = reinterpret_cast<const float4*>(xs + c * a.H + v * EPV);
              float4 x0 = xp[0];
              float t = acc[c];
              t = fmaf(wf[0], x0.x, t); t = fmaf(wf[1], x0.y, t);
              t = fmaf(wf[2], x0.z, t); t = fmaf(wf[3], x0.w, t);
              if (EPV == 8) {
                float4 x1 = xp[1];
                t = fmaf(wf[4], x1.x, t); t = fmaf(wf[5], x1.y, t);
                t = fmaf(wf[6], x1.z, t); t = fmaf(wf[7], x1.w, t);
              }
              acc[c] = t;
            }
          }
        }
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] = warp_sum(acc[c]);

      // ---- per-row epilogue: lane c owns column c0 + c
      const int j = r - seg * a.S;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        if (lane == c && c0 + c < a.C) {
          if (EPI == EPI_FC) {
            const float pre = acc[c] + to_f32(reinterpret_cast<const TW*>(a.bias)[(size_t)seg * a.H + j]);
            const float silu = pre / (1.f + expf(-pre));
            a.z[((size_t)(c0 + c) * a.nseg + seg) * a.H + j] = xs[c * a.H + j] + silu;
          } else if (EPI == EPI_TOPK) {
            rowbuf[c * kRowBuf + (r - r0)] = acc[c];
          } else {
            soft_push(soft, acc[c], a.id_off + j, typical, a.inv_temp);
          }
        }
      }
    }

    // ---- end of piece: warp c picks the top-kn rows of column c
    if (EPI == EPI_TOPK) {
      __syncthreads();
      if (warp < NC && c0 + warp < a.C) {
        const int c = warp;
        float lv[KMAX];
        int li[KMAX];
        list_reset(lv, li);
        for (int e = lane; e < r1 - r0; e += 32)
          list_insert(lv, li, kn, rowbuf[c * kRowBuf + e], a.id_off + r0 + e - seg * a.S);
        const size_t base = ((size_t)(cta * kMaxPieces + piece) * a.C + (c0 + c)) * a.kmax;
        warp_select(lv, li, kn, a.kmax, a.cand_val + base, a.cand_idx + base, INT_MAX);
      }
      if (threadIdx.x == 0 && blockIdx.y == 0) a.cand_seg[cta * kMaxPieces + piece] = seg;
    }
    r0 = r1;
  }
  if (EPI == EPI_TOPK && threadIdx.x == 0 && blockIdx.y == 0)
    for (int p = piece; p < kMaxPieces; ++p) a.cand_seg[cta * kMaxPieces + p] = -1;

  if (EPI == EPI_VERIFY) {
    if (lane < NC) wsoft[warp][lane] = soft;
    __syncthreads();
    if (warp == 0 && lane < NC && c0 + lane < a.C) {
      SoftState m = wsoft[0][lane];
      for (int w = 1; w < kWarps; ++w) m = soft_merge(m, wsoft[w][lane], typical, a.inv_temp);
      const size_t pi = (size_t)cta * a.C + c0 + lane;
      a.part[pi * 3 + 0] = m.m;
      a.part[pi * 3 + 1] = m.z;
      a.part[pi * 3 + 2] = m.s;
      a.part_idx[pi] = m.mi;
    }
  }
  if (EPI != EPI_VERIFY) return;  // top-k candidates are merged by topk_merge_kernel

  // ---- last CTA merges every CTA's partial result
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int total = gridDim.x * gridDim.y;
    s_last = (atomicAdd(a.ticket, 1) == total - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int nctas = gridDim.x;

  if (EPI == EPI_VERIFY) {
    for (int c = warp; c < a.C; c += kWarps) {
      SoftState m;
      m.m = -INFINITY;
      m.z = 0.f;
      m.s = 0.f;
      m.mi = INT_MAX;
      for (int blk = lane; blk < nctas; blk += 32) {
        const size_t pi = (size_t)blk * a.C + c;
        SoftState o;
        o.m = a.part[pi * 3 + 0];
        o.z = a.part[pi * 3 + 1];
        o.s = a.part[pi * 3 + 2];
        o.mi = a.part_idx[pi];
        m = soft_merge(m, o, typical, a.inv_temp);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        SoftState t;
        t.m = __shfl_xor_sync(0xffffffffu, m.m, o);
        t.z = __shfl_xor_sync(0xffffffffu, m.z, o);
        t.s = __shfl_xor_sync(0xffffffffu, m.s, o);
        t.mi = __shfl_xor_sync(0xffffffffu, m.mi, o);
        m = soft_merge(m, t, typical, a.inv_temp);
      }
      if (lane == 0 && a.soft_out) {
        a.soft_out[c] = make_float4(m.m, m.z, m.s, __int_as_float(m.mi));
      } else if (lane == 0) {
        a.node_argmax[c] = m.mi;
        a.node_maxlogit[c] = m.m;
        if (typical) {
          const float lz = logf(m.z);
          if (a.node_lse) a.node_lse[c] = m.m * a.inv_temp + lz;
          if (a.node_entropy) a.node_entropy[c] = lz - m.s / m.z;
        }
      }
    }
  }
  if (threadIdx.x == 0) *a.ticket = 0;  // ready for the next call
}

// Final per-head top-k: one warp per (segment, column) folds the candidate
// lists of the CTAs whose row range touched the segment (loads spread over the
// lanes), then picks the best kn with warp_select.
template <int KM>
__global__ void __launch_bounds__(256) topk_merge_kernel(RowArgs a, int nctas) {
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_trigger();
  pdl_wait();
  if (pair >= a.nseg * a.C) return;
  const int seg = pair / a.C, c = pair - seg * a.C;
  const int kn = kept_of(a, seg);
  const int b_lo = (int)(((long long)seg * a.S) / a.rpc);
  const int b_hi = min(nctas - 1, (int)(((long long)(seg + 1) * a.S - 1) / a.rpc));
  float lv[KM];
  int li[KM];
  list_reset(lv, li);
  const int n_slots = (b_hi - b_lo + 1) * kMaxPieces;
  for (int sl = lane; sl < n_slots; sl += 32) {
    const int blk = b_lo + sl / kMaxPieces, p = sl % kMaxPieces;
    if (a.cand_seg[blk * kMaxPieces + p] != seg) continue;
    const size_t base = ((size_t)(blk * kMaxPieces + p) * a.C + c) * a.kmax;
    for (int i = 0; i < kn; ++i) list_insert(lv, li, kn, a.cand_val[base + i], a.cand_idx[base + i]);
  }
  const size_t o = ((size_t)c * a.nseg + seg) * a.kmax;
  warp_select(lv, li, kn, a.kmax, a.out_val + o, a.out_idx + o, -1);
}

// --------------------------------------------------------------- launchers --
// rows per CTA so that a grid of `want` CTAs covers R rows with no CTA
// spanning more than kMaxPieces segments of S rows
static void partition(int R, int S, int want, int max_rows, int min_rows, int* ctas, int* rpc) {
  if (want > kMaxStreamCtas) want = kMaxStreamCtas;
  if (want < 1) want = 1;
  int r = (R + want - 1) / want;
  if (r < min_rows) r = min_rows;
  if (r > max_rows) r = max_rows;
  const int cap = (kMaxPieces - 1) * S;
  if (r > cap) r = cap;
  *rpc = r;
  *ctas = (R + r - 1) / r;
}

// Launches one persistent grid of (SM count x resident CTAs per SM) CTAs per
// column tile; the grid size comes from the occupancy of the instance.
template <typename TW, typename TX, int EPI>
static int launch_nc(RowArgs a, int sm_count, int nc, int ctiles, cudaStream_t st, int* ctas_out = nullptr,
                     int* rpc_out = nullptr) {
  const size_t smem = (size_t)nc * a.H * sizeof(float) + (EPI == EPI_TOPK ? (size_t)nc * kRowBuf * sizeof(float) : 0);
  cudaError_t e = cudaSuccess;
#define MEDUSA_LAUNCH_NC(N)                                                                                 \
  case N: {                                                                                                 \
    auto k = stream_rows_kernel<TW, TX, N, EPI>;                                                            \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);                    \
    int occ = 0;                                                                                            \
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, smem);       \
    if (e == cudaSuccess) {                                                                                 \
      int ctas = 0;                                                                                         \
      /* epilogues with a merge take at least four rows per warp: a small weight then */                   \
      /* takes tens of CTAs instead of hundreds of one-row CTAs whose partials are merged one by one */   \
      partition(a.R, a.S, sm_count * (occ > 0 ? occ : 1), EPI == EPI_TOPK ? kRowBuf : (1 << 30),           \
                EPI == EPI_FC ? 1 : 4 * kWarps, &ctas, &a.rpc);                                             \
      if (ctas > kMaxStreamCtas) return (int)cudaErrorInvalidConfiguration;                                 \
      e = launch_k(k, dim3(ctas, ctiles), dim3(kThreads), smem, st, EPI != EPI_FC, a);                      \
      if (ctas_out) *ctas_out = ctas;                                                                       \
      if (rpc_out) *rpc_out = a.rpc;                                                                        \
      if (e == cudaSuccess && EPI == EPI_TOPK && !ctas_out) { /* else the caller merges */                  \
        const unsigned mg = (unsigned)((a.nseg * a.C + 7) / 8);                                             \
        if (a.kmax <= 4) e = launch_k(topk_merge_kernel<4>, dim3(mg), dim3(256), 0, st, true, a, ctas);     \
        else e = launch_k(topk_merge_kernel<KMAX>, dim3(mg), dim3(256), 0, st, true, a, ctas);              \
      }                                                                                                     \
    }                                                                                                       \
    break;                                                                                                  \
  }
  switch (nc) {
    MEDUSA_LAUNCH_NC(1)
    MEDUSA_LAUNCH_NC(2)
    MEDUSA_LAUNCH_NC(4)
    MEDUSA_LAUNCH_NC(8)
    default:
      return (int)cudaErrorInvalidValue;
  }
#undef MEDUSA_LAUNCH_NC
  return (int)e;
}

// Final top-k merge for candidates written by any streaming kernel.
// CTA c of that kernel covered work units [c * rpc, (c + 1) * rpc), S units per head.
int launch_topk_merge(const Plan& p, int32_t* topk_idx, float* topk_val, uint8_t* ws, int ctas, int rpc, int S,
                      cudaStream_t st) {
  RowArgs a{};
  a.R = p.K * S;
  a.S = S;
  a.H = p.H;
  a.C = p.B;
  a.rpc = rpc;
  a.nseg = p.K;
  a.kmax = p.kmax;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.topk_n[k] = p.topk_n[k];
  a.cand_val = reinterpret_cast<float*>(ws + p.off_cand_val);
  a.cand_idx = reinterpret_cast<int*>(ws + p.off_cand_idx);
  a.cand_seg = reinterpret_cast<int*>(ws + p.off_cand_seg);
  a.out_idx = topk_idx;
  a.out_val = topk_val;
  const unsigned mg = (unsigned)((a.nseg * a.C + 7) / 8);
  if (a.kmax <= 4) return (int)launch_k(topk_merge_kernel<4>, dim3(mg), dim3(256), 0, st, true, a, ctas);
  return (int)launch_k(topk_merge_kernel<KMAX>, dim3(mg), dim3(256), 0, st, true, a, ctas);
}

int launch_fc(const Plan& p, const void* h, const void* W1, const void* b1, uint8_t* ws, cudaStream_t st) {
  RowArgs a{};
  a.W = W1;
  a.x = h;
  a.x_cs = p.H;
  a.x_ss = 0;
  a.R = p.K * p.H;
  a.S = p.H;
  a.H = p.H;
  a.C = p.B;
  a.nseg = p.K;
  a.ws = ws;
  a.bias = b1;
  a.z = reinterpret_cast<float*>(ws + p.off_z);
  if (p.bf16) return launch_nc<__nv_bfloat16, __nv_bfloat16, EPI_FC>(a, p.sm_count, p.fc_nc, p.fc_ctiles, st);
  return launch_nc<float, float, EPI_FC>(a, p.sm_count, p.fc_nc, p.fc_ctiles, st);
}

// ctas / rpc non-null: the candidates stay in the workspace for the caller's
// merge (the grid and rows per CTA are reported); otherwise the top-k merge
// is launched here
int launch_proj_topk(const Plan& p, const void* W2, int32_t* topk_idx, float* topk_val, uint8_t* ws,
                     cudaStream_t st, int* ctas, int* rpc) {
  RowArgs a{};
  a.W = W2;
  a.x = ws + p.off_z;
  a.x_cs = (long long)p.K * p.H;
  a.x_ss = p.H;
  a.R = p.K * p.Vs;
  a.S = p.Vs;
  a.id_off = p.v0;
  a.H = p.H;
  a.C = p.B;
  a.nseg = p.K;
  a.ws = ws;
  a.ticket = reinterpret_cast<int*>(ws) + TICKET_PROJ;
  a.kmax = p.kmax;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.topk_n[k] = p.topk_n[k];
  a.cand_val = reinterpret_cast<float*>(ws + p.off_cand_val);
  a.cand_idx = reinterpret_cast<int*>(ws + p.off_cand_idx);
  a.cand_seg = reinterpret_cast<int*>(ws + p.off_cand_seg);
  a.out_idx = topk_idx;
  a.out_val = topk_val;
  if (p.bf16) return launch_nc<__nv_bfloat16, float, EPI_TOPK>(a, p.sm_count, p.pj_nc, p.pj_ctiles, st, ctas, rpc);
  return launch_nc<float, float, EPI_TOPK>(a, p.sm_count, p.pj_nc, p.pj_ctiles, st, ctas, rpc);
}

int launch_verify_rows(const Plan& p, const void* attn_out, const void* lm_head, int32_t* node_argmax,
                       float* node_maxlogit, float* node_lse, float* node_entropy, uint8_t* ws, cudaStream_t st,
                       float4* soft_out) {
  RowArgs a{};
  a.W = lm_head;
  a.x = attn_out;
  a.x_cs = p.H;
  a.x_ss = 0;
  a.R = p.Vs;
  a.S = p.Vs;
  a.id_off = p.v0;
  a.soft_out = soft_out;
  a.H = p.H;
  a.C = p.B * p.T;
  a.nseg = 1;
  a.ws = ws;
  a.ticket = reinterpret_cast<int*>(ws) + TICKET_VERIFY;
  a.typical = p.typical ? 1 : 0;
  a.inv_temp = p.typical ? 1.f / p.temperature : 1.f;
  a.part = reinterpret_cast<float*>(ws + p.off_vf_part);
  a.part_idx = reinterpret_cast<int*>(ws + p.off_vf_idx);
  a.node_argmax = node_argmax;
  a.node_maxlogit = node_maxlogit;
  a.node_lse = node_lse;
  a.node_entropy = node_entropy;
  if (p.bf16) return launch_nc<__nv_bfloat16, __nv_bfloat16, EPI_VERIFY>(a, p.sm_count, p.vf_nc, p.vf_ctiles, st);
  return launch_nc<float, float, EPI_VERIFY>(a, p.sm_count, p.vf_nc, p.vf_ctiles, st);
}

}  // namespace medusa
