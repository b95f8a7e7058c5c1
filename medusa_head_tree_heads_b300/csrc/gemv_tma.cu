// Small-batch weight streaming for the Medusa heads ("Medusa Heads", "Come le
// teste prevedono i token successivi": each head is a residual SiLU layer,
// z = h + SiLU(W1 h + b1), then a vocabulary projection W2 z; "Attenzione
// sull'albero e accettazione": the best tokens of each head form the tree).
//
//   out[c][r] = W[r] . x[c, seg(r)],  r < R rows of H bf16, c < NC <= 4 columns
//   EPI_FC:   z[c][seg][j] = h[c][j] + SiLU(out + b1[seg][j])      (W = W1)
//   EPI_TOPK: per-CTA top-k candidates of every (segment, column)  (W = W2)
//
// At batch <= 4 this is a pure HBM stream, so the kernel is built to keep
// bytes in flight with almost no instruction overhead:
//   * a persistent grid, one CTA per SM, splits the rows into equal
//     contiguous ranges; a CTA's rows are one contiguous byte range of W;
//   * a producer warp streams it with 1-D bulk copies (cp.async.bulk,
//     mbarrier completion) through an S-stage shared-memory ring of RB rows
//     per stage (a stage never crosses a segment boundary);
//   * 8 consumer warps split the columns: thread t owns 16-byte vectors
//     t, t+256, ... of every row, holds the matching x values in registers
//     (fp32), and reads the weights from shared memory conflict-free;
//   * one warp reduction and a named barrier per stage turn the 256 partial
//     sums of each row into the row's value.
// The projection's per-CTA candidates are merged by topk_merge_kernel.
#include <limits.h>

#include "internal.cuh"
#include "tc.cuh"

namespace medusa {

constexpr int GT_RB = 4;               // rows per stage
constexpr int GT_CONS = 256;           // consumer threads (8 warps)
constexpr int GT_THREADS = GT_CONS + 32;  // + producer warp
constexpr uint64_t GT_WAIT_NS = 20ull * 1000 * 1000;
constexpr int GT_ROWBUF = 2048;        // rows per CTA (top-k row values kept in shared memory)
constexpr int GT_GROUP = 8;            // max stages per reduction group (32 values per thread)

struct GtArgs {
  const __nv_bfloat16* W;  // [R][H]
  const void* x;           // fp32 (x_f32) or bf16: x(c, seg, j) = x[c * x_cs + seg * x_ss + j]
  int x_f32;
  long long x_cs, x_ss;
  int R, S, H, C, nseg, rpc, stages;
  uint8_t* ws;
  // EPI_FC
  const __nv_bfloat16* bias;  // [nseg][H]
  const __nv_bfloat16* hres;  // [C][H] residual input
  float* z;                   // [C][nseg][H]
  // EPI_TOPK
  int kmax;
  int topk_n[MEDUSA_MAX_HEADS];
  float* cand_val;
  int* cand_idx;
  int* cand_seg;
};

template <int VPL, int NC>
__device__ __forceinline__ void load_x(const GtArgs& a, int seg, int t, float (&xr)[NC][VPL][8]) {
  const int nvec = a.H / 8;
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = t + GT_CONS * i;
#pragma unroll
      for (int e = 0; e < 8; ++e) xr[c][i][e] = 0.f;
      if (v < nvec && c < a.C) {
        const long long off = (long long)c * a.x_cs + (long long)seg * a.x_ss + (long long)v * 8;
        if (a.x_f32) {
          const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.x) + off);
          const float4 p0 = p[0], p1 = p[1];
          xr[c][i][0] = p0.x; xr[c][i][1] = p0.y; xr[c][i][2] = p0.z; xr[c][i][3] = p0.w;
          xr[c][i][4] = p1.x; xr[c][i][5] = p1.y; xr[c][i][6] = p1.z; xr[c][i][7] = p1.w;
        } else {
          const uint4 p = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.x) + off);
          xr[c][i][0] = bf16_lo(p.x); xr[c][i][1] = bf16_hi(p.x);
          xr[c][i][2] = bf16_lo(p.y); xr[c][i][3] = bf16_hi(p.y);
          xr[c][i][4] = bf16_lo(p.z); xr[c][i][5] = bf16_hi(p.z);
          xr[c][i][6] = bf16_lo(p.w); xr[c][i][7] = bf16_hi(p.w);
        }
      }
    }
}

__device__ __forceinline__ int gt_kept(const GtArgs& a, int seg) {
  int n = 1;
#pragma unroll
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k)
    if (k == seg) n = a.topk_n[k];
  return n;
}

// stage schedule shared by producer and consumers: rows [row, row + n) of segment seg
__device__ __forceinline__ void next_stage(const GtArgs& a, int r_end, int& row, int& n, int& seg) {
  seg = row / a.S;
  const int seg_end = min(r_end, (seg + 1) * a.S);
  n = min(GT_RB, seg_end - row);
}

template <int VPL, int NC, int EPI>
__global__ void __launch_bounds__(GT_THREADS, 1) gemv_tma_kernel(GtArgs a) {
  extern __shared__ uint8_t gt_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gt_raw) + 127) & ~uintptr_t(127));
  const int S = a.stages;
  const size_t row_bytes = (size_t)a.H * 2;
  const size_t stage_bytes = GT_RB * row_bytes;
  float* rowbuf = reinterpret_cast<float*>(smem + (size_t)S * stage_bytes);  // [NC][GT_ROWBUF] (EPI_TOPK)
  float* red = rowbuf + (EPI == 1 ? NC * GT_ROWBUF : 0);                   // [2][8 warps][32 values]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 2 * 8 * 32);
  uint64_t* empty = full + S;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r_begin = blockIdx.x * a.rpc;
  const int r_end = min(a.R, r_begin + a.rpc);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 8);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();

  if (warp == 8) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t k = 0;
      bool ok = true;
      for (int row = r_begin; row < r_end; ++k) {
        int n, seg;
        next_stage(a, r_end, row, n, seg);
        const int s = k % S;
        const uint32_t ph = (k / S) & 1u;
        if (!tc::mbar_try_wait(&empty[s], ph ^ 1u)) {
          const uint64_t t0 = tc::globaltimer_ns();
          while (!tc::mbar_try_wait(&empty[s], ph ^ 1u)) {
            if (*abort_flag || tc::globaltimer_ns() - t0 > GT_WAIT_NS) {
              if (!*abort_flag) set_error(a.ws, MEDUSA_ERR_TIMEOUT);
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        const uint32_t bytes = (uint32_t)(n * row_bytes);
        tc::mbar_arrive_expect_tx(&full[s], bytes);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                tc::smem_u32(smem + (size_t)s * stage_bytes)),
            "l"(a.W + (size_t)row * a.H), "r"(bytes), "r"(tc::smem_u32(&full[s]))
            : "memory");
        row += n;
      }
      if (!ok) {  // let the copies already issued land before the CTA leaves
        const uint32_t first = k > (uint32_t)S ? k - S : 0;
        for (uint32_t ki = first; ki < k; ++ki) {
          const uint64_t t0 = tc::globaltimer_ns();
          while (!tc::mbar_try_wait(&full[ki % S], (ki / S) & 1u) && tc::globaltimer_ns() - t0 < GT_WAIT_NS) {
          }
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  // (the producer streams weights, which no kernel writes, before the
  // preceding kernel has finished; x, z and the outputs wait for it)
  pdl_wait();
  const int nvec = a.H / 8;
  float xr[NC][VPL][8];
  int cur_seg = -1;
  uint32_t k = 0;           // stage counter (same schedule as the producer)
  int row = r_begin;
  int piece = 0, piece_row0 = r_begin, piece_seg = r_begin / a.S;
  int* grp_row = reinterpret_cast<int*>(full + 2 * S) + 4;  // [GT_GROUP] first row of each slot (-1: none)
  int* grp_n = grp_row + GT_GROUP;                           // [GT_GROUP] rows in each slot
  bool aborted = false;
  constexpr int GR = 32 / NC;           // group rows per column
  constexpr int GSLOT = GR / GT_RB;     // stages per group
  for (int grp = 0; row < r_end && !aborted; ++grp) {
    // ---- a group: GSLOT stages of GT_RB rows; acc[c * GR + r] holds this
    // thread's partial sum of group row r (GR = 32 / NC rows) for column c
    float acc[32];
#pragma unroll
    for (int g = 0; g < 32; ++g) acc[g] = 0.f;
#pragma unroll
    for (int slot = 0; slot < GSLOT; ++slot) {
      int n = 0, seg = cur_seg;
      if (row < r_end) next_stage(a, r_end, row, n, seg);
      if (tid == 0) {
        grp_row[slot] = n > 0 ? row : -1;
        grp_n[slot] = n;
      }
      if (n > 0) {
        if (seg != cur_seg) {  // uniform: every consumer reloads its x slice
          load_x<VPL, NC>(a, seg, tid, xr);
          cur_seg = seg;
        }
        const int s = k % S;
        const uint32_t ph = (k / S) & 1u;
        bool ok = tc::mbar_try_wait(&full[s], ph);
        if (!ok) {
          const uint64_t t0 = tc::globaltimer_ns();
          while (!(ok = tc::mbar_try_wait(&full[s], ph))) {
            if (*abort_flag) break;
            if (tc::globaltimer_ns() - t0 > GT_WAIT_NS) {
              set_error(a.ws, MEDUSA_ERR_TIMEOUT);
              *abort_flag = 1;
              break;
            }
          }
        }
        if (ok) {
          const uint8_t* st = smem + (size_t)s * stage_bytes;
#pragma unroll
          for (int rr = 0; rr < GT_RB; ++rr) {
            uint4 w[VPL];
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
              const int v = tid + GT_CONS * i;
              w[i] = (rr < n && v < nvec) ? *reinterpret_cast<const uint4*>(st + rr * row_bytes + (size_t)v * 16)
                                          : make_uint4(0u, 0u, 0u, 0u);
            }
            // VPL * NC independent chains of 8 FMAs for this row (rows interleave after unrolling)
            float part[VPL][NC];
#pragma unroll
            for (int i = 0; i < VPL; ++i)
#pragma unroll
              for (int c = 0; c < NC; ++c) part[i][c] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
              for (int i = 0; i < VPL; ++i) {
                const uint32_t wv = e < 2 ? w[i].x : e < 4 ? w[i].y : e < 6 ? w[i].z : w[i].w;
                const float wf = (e & 1) ? bf16_hi(wv) : bf16_lo(wv);
#pragma unroll
                for (int c = 0; c < NC; ++c) part[i][c] = fmaf(wf, xr[c][i][e], part[i][c]);
              }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              float t = 0.f;
#pragma unroll
              for (int i = 0; i < VPL; ++i) t += part[i][c];
              acc[c * GR + slot * GT_RB + rr] = t;
            }
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[s]);  // this warp has read the stage
        ++k;
        row += n;
      }
    }
    // ---- butterfly transpose-reduce over the 32 lanes: lane l ends with the
    // warp's partial of value l (column l / GR, group row l % GR); 31 exchanges
#pragma unroll
    for (int step = 0; step < 5; ++step) {
      const int o = 16 >> step, half = 16 >> step;
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = up ? acc[i] : acc[i + half];
        const float keep = up ? acc[i + half] : acc[i];
        acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    const int par = grp & 1;
    red[(par * 8 + warp) * 32 + lane] = acc[0];
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (*abort_flag) aborted = true;
    // ---- row values: thread t < 32 finishes value t (column t / GR, group row t % GR)
    if (!aborted && tid < 32) {
      const int c = tid / GR, gr = tid % GR;
      const int r0 = grp_row[gr / GT_RB];
      if (r0 >= 0 && (gr % GT_RB) < grp_n[gr / GT_RB] && c < a.C) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) t += red[(par * 8 + w) * 32 + tid];
        const int r = r0 + gr % GT_RB;
        const int seg = r / a.S, j = r - seg * a.S;
        if (EPI == 0) {
          const float pre = t + __bfloat162float(a.bias[(size_t)seg * a.H + j]);
          const float silu = pre / (1.f + expf(-pre));
          a.z[((size_t)c * a.nseg + seg) * a.H + j] = __bfloat162float(a.hres[(size_t)c * a.H + j]) + silu;
        } else {
          rowbuf[c * GT_ROWBUF + (r - r_begin)] = t;
        }
      }
    }
    // ---- top-k of every segment piece that ended in (or before) this group
    if (EPI == 1) {
      const int seg_now = row < r_end ? row / a.S : -1;
      if (seg_now != piece_seg) {
        asm volatile("bar.sync 1, 256;" ::: "memory");  // rowbuf complete
        // pieces [piece_row0, end) of piece_seg, and any whole segment in between (none: rpc <= S)
        const int end = row < r_end ? seg_now * a.S : r_end;
        if (!aborted && warp < NC && warp < a.C) {
          const int kn = gt_kept(a, piece_seg);
          float lv[MEDUSA_MAX_TOPK];
          int li[MEDUSA_MAX_TOPK];
#pragma unroll
          for (int i = 0; i < MEDUSA_MAX_TOPK; ++i) {
            lv[i] = -INFINITY;
            li[i] = INT_MAX;
          }
          for (int e = lane; e < end - piece_row0; e += 32) {
            float cv = rowbuf[warp * GT_ROWBUF + (piece_row0 - r_begin) + e];
            int ci = piece_row0 + e - piece_seg * a.S;
#pragma unroll
            for (int i = 0; i < MEDUSA_MAX_TOPK; ++i) {  // compare-and-swap insertion
              const bool sw = (i < kn) && better(cv, ci, lv[i], li[i]);
              const float ov = lv[i];
              const int oi = li[i];
              lv[i] = sw ? cv : ov;
              li[i] = sw ? ci : oi;
              cv = sw ? ov : cv;
              ci = sw ? oi : ci;
            }
          }
          const size_t base = ((size_t)(blockIdx.x * kMaxPieces + piece) * a.C + warp) * a.kmax;
          for (int rnk = 0; rnk < a.kmax; ++rnk) {
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
            if (bi != INT_MAX && lv[0] == bv && li[0] == bi) {
#pragma unroll
              for (int i = 0; i < MEDUSA_MAX_TOPK - 1; ++i) {
                lv[i] = lv[i + 1];
                li[i] = li[i + 1];
              }
              lv[MEDUSA_MAX_TOPK - 1] = -INFINITY;
              li[MEDUSA_MAX_TOPK - 1] = INT_MAX;
            }
            if (lane == 0) {
              const bool live = rnk < kn && bi != INT_MAX;
              a.cand_val[base + rnk] = live ? bv : -INFINITY;
              a.cand_idx[base + rnk] = live ? bi : INT_MAX;
            }
          }
        }
        if (tid == 0) a.cand_seg[blockIdx.x * kMaxPieces + piece] = aborted ? -1 : piece_seg;
        ++piece;
        piece_row0 = end;
        piece_seg = seg_now;
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // grp_row / grp_n are rewritten by the next group
  }
  if (EPI == 1 && tid == 0)
    for (int p = piece; p < kMaxPieces; ++p) a.cand_seg[blockIdx.x * kMaxPieces + p] = -1;
}

// ------------------------------------------------------------------- host --
// Returns cudaErrorNotSupported when the shape is outside this kernel's range
// (the caller then uses the general streaming kernel).
template <int EPI>
static int gemv_tma_launch(GtArgs a, int sm_count, int nc, cudaStream_t st, int* ctas_out, int max_stages = 8) {
  const int nvec = a.H / 8;
  const int vpl = (nvec + GT_CONS - 1) / GT_CONS;
  if (vpl > 4 || nc > 4 || a.C > nc) return (int)cudaErrorNotSupported;
  // one CTA per SM; every CTA owns at most GT_ROWBUF rows and 2 segment pieces
  int ctas = sm_count;
  int rpc = (a.R + ctas - 1) / ctas;
  if (EPI == 1 && rpc > GT_ROWBUF) return (int)cudaErrorNotSupported;
  if (rpc > a.S) return (int)cudaErrorNotSupported;  // pieces per CTA stay <= 2
  ctas = (a.R + rpc - 1) / rpc;
  if (ctas > kMaxStreamCtas) return (int)cudaErrorNotSupported;
  a.rpc = rpc;
  const size_t stage = (size_t)GT_RB * a.H * 2;
  const size_t fixed = 128 + (EPI == 1 ? (size_t)nc * GT_ROWBUF * 4 : 0) + 2 * 8 * 32 * 4 + 512;
  int S = (int)((220 * 1024 - fixed) / stage);
  if (S > max_stages) S = max_stages;
  if (S < 2) return (int)cudaErrorNotSupported;
  a.stages = S;
  const size_t smem = fixed + (size_t)S * stage;
  void (*k)(GtArgs) = nullptr;
#define GT_PICK(V, N) \
  if (vpl == V && nc == N) k = gemv_tma_kernel<V, N, EPI>;
  GT_PICK(1, 1) GT_PICK(2, 1) GT_PICK(3, 1) GT_PICK(4, 1)
  GT_PICK(1, 2) GT_PICK(2, 2) GT_PICK(3, 2) GT_PICK(4, 2)
  GT_PICK(1, 4) GT_PICK(2, 4) GT_PICK(3, 4) GT_PICK(4, 4)
#undef GT_PICK
  if (!k) return (int)cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  // the whole unified L1/shared array as shared memory, so that a kernel
  // co-scheduled on the same SM (the tree attention) finds room beside this one
  e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return (int)e;
  if (ctas_out) *ctas_out = ctas;
  // programmatic dependent launch for both: the producer streams weights
  // (written by no kernel) at once; x, z and the outputs wait for the grid before
  return (int)launch_k(k, dim3(ctas), dim3(GT_THREADS), smem, st, true, a);
}

static int gt_nc(int B) { return B <= 1 ? 1 : (B <= 2 ? 2 : 4); }

bool gemv_tma_supported(const Plan& p) {
  if (!p.bf16 || p.B > 4 || p.H / 8 > 4 * GT_CONS) return false;
  const int rpc_fc = (p.K * p.H + p.sm_count - 1) / p.sm_count;
  const int rpc_pj = (p.K * p.V + p.sm_count - 1) / p.sm_count;
  return rpc_fc <= p.H && rpc_pj <= p.V && rpc_pj <= GT_ROWBUF;
}

int launch_fc_tma(const Plan& p, const void* h, const void* W1, const void* b1, uint8_t* ws, cudaStream_t st) {
  GtArgs a{};
  a.W = reinterpret_cast<const __nv_bfloat16*>(W1);
  a.x = h;
  a.x_f32 = 0;
  a.x_cs = p.H;
  a.x_ss = 0;
  a.R = p.K * p.H;
  a.S = p.H;
  a.H = p.H;
  a.C = p.B;
  a.nseg = p.K;
  a.ws = ws;
  a.bias = reinterpret_cast<const __nv_bfloat16*>(b1);
  a.hres = reinterpret_cast<const __nv_bfloat16*>(h);
  a.z = reinterpret_cast<float*>(ws + p.off_z);
  return gemv_tma_launch<0>(a, p.sm_count, gt_nc(p.B), st, nullptr);
}

int launch_topk_merge(const Plan& p, int32_t* topk_idx, float* topk_val, uint8_t* ws, int ctas, int rpc, int S,
                      cudaStream_t st);

// The projection kernel alone (its candidates merged later by launch_topk_merge);
// max_stages bounds the shared ring so another kernel can share the SM.
int launch_proj_tma_only(const Plan& p, const void* W2, uint8_t* ws, cudaStream_t st, int max_stages, int* ctas,
                         int* rpc) {
  GtArgs a{};
  a.W = reinterpret_cast<const __nv_bfloat16*>(W2);
  a.x = ws + p.off_z;
  a.x_f32 = 1;
  a.x_cs = (long long)p.K * p.H;
  a.x_ss = p.H;
  a.R = p.K * p.V;
  a.S = p.V;
  a.H = p.H;
  a.C = p.B;
  a.nseg = p.K;
  a.ws = ws;
  a.kmax = p.kmax;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.topk_n[k] = p.topk_n[k];
  a.cand_val = reinterpret_cast<float*>(ws + p.off_cand_val);
  a.cand_idx = reinterpret_cast<int*>(ws + p.off_cand_idx);
  a.cand_seg = reinterpret_cast<int*>(ws + p.off_cand_seg);
  *rpc = (a.R + p.sm_count - 1) / p.sm_count;
  return gemv_tma_launch<1>(a, p.sm_count, gt_nc(p.B), st, ctas, max_stages);
}

int launch_proj_tma(const Plan& p, const void* W2, int32_t* topk_idx, float* topk_val, uint8_t* ws,
                    cudaStream_t st) {
  GtArgs a{};
  a.W = reinterpret_cast<const __nv_bfloat16*>(W2);
  a.x = ws + p.off_z;
  a.x_f32 = 1;
  a.x_cs = (long long)p.K * p.H;
  a.x_ss = p.H;
  a.R = p.K * p.V;
  a.S = p.V;
  a.H = p.H;
  a.C = p.B;
  a.nseg = p.K;
  a.ws = ws;
  a.kmax = p.kmax;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.topk_n[k] = p.topk_n[k];
  a.cand_val = reinterpret_cast<float*>(ws + p.off_cand_val);
  a.cand_idx = reinterpret_cast<int*>(ws + p.off_cand_idx);
  a.cand_seg = reinterpret_cast<int*>(ws + p.off_cand_seg);
  int ctas = 0;
  int e = gemv_tma_launch<1>(a, p.sm_count, gt_nc(p.B), st, &ctas);
  if (e) return e;
  const int rpc = (a.R + p.sm_count - 1) / p.sm_count;
  return launch_topk_merge(p, topk_idx, topk_val, ws, ctas, rpc, p.V, st);
}

}  // namespace medusa
