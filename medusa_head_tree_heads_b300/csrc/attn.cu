// Tree attention, one pass over the KV cache and the tree ("Medusa Heads",
// "Attenzione sull'albero e accettazione": every candidate token is appended
// to the input at once and a mask lets each see only its ancestors;
// "Tetes de decodage Medusa", "Plongee profonde": the whole tree is verified
// in one pass with a tree attention mask).
//
// For sequence b, kv head g and query row r = node * G + (q head - g*G):
//   o = sum_j softmax_j(q . k_j / sqrt(Dh)) v_j,
//   j over cache rows [0, L) and tree nodes j with bit j of the node's mask row.
//
// CUDA-core version: a CTA owns up to 16 query rows (2 for small grids) of one (b, g); its 8
// warps split the group's keys (cache tiles, then tree tiles masked by the
// rows' mask words) between them, tile w, w + 8, ... for warp w, each warp
// keeping an fp32 online softmax per row over its own tiles in registers and
// its own K/V tile in shared memory (no CTA-wide barrier in the key loop).
// The 8 partial states of every row are joined at the end through shared
// memory.  No partial results leave the CTA, so no combine launch.  A tile is
// 32 keys for head dim 64 (lane = key) and 16 keys for head dim 128.
#include "internal.cuh"

namespace medusa {

constexpr int AF_ROWS = 16;   // query rows per CTA
constexpr int AF_ROWS_FEW = 2;  // ... when 16 would leave most SMs idle
constexpr int AF_WARPS = 8;

struct AttnArgs {
  const void *q, *kt, *vt, *kc, *vc;
  TreeDims td;           // the tree's parent table: each CTA builds its rows' ancestor masks from it
  size_t smem_floats;    // the float area of dynamic shared memory; the rows' masks follow it
  void* out;             // [B][T][H]
  int B, T, W, Hq, Hkv, G, L, Lc, H;
  float qscale;  // log2(e) / sqrt(Dh)
  const int32_t* lens;  // [B] per-sequence cache lengths, or null (L for all)
  uint8_t* ws;
};

template <int DH>
constexpr int af_keys() { return DH == 64 ? 32 : 16; }
template <int DH, int ROWS>
constexpr size_t af_smem_floats() {  // queries + per warp one K tile (padded rows) and one V tile
  return (size_t)ROWS * DH + (size_t)AF_WARPS * af_keys<DH>() * (2 * DH + 1);
}

template <typename TT, int DH, int ROWS>
__global__ void __launch_bounds__(AF_WARPS * 32) tree_attn_kernel(AttnArgs a) {
  constexpr int DPL = DH / 32;      // output dims per lane
  constexpr int KT = af_keys<DH>();  // keys per tile
  extern __shared__ float4 at_smem[];
  float* qs = reinterpret_cast<float*>(at_smem);  // [ROWS][DH]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* ks = qs + ROWS * DH + (size_t)warp * KT * (2 * DH + 1);  // this warp's [KT][DH + 1]
  float* vs = ks + KT * (DH + 1);                                     // this warp's [KT][DH]
  const int g = blockIdx.y, b = blockIdx.z;
  const int row0 = blockIdx.x * ROWS;
  const int nrows = a.T * a.G;
  const TT* Q = reinterpret_cast<const TT*>(a.q);
  uint32_t* mrow = reinterpret_cast<uint32_t*>(reinterpret_cast<float*>(at_smem) + a.smem_floats);  // [ROWS][W]
  pdl_trigger();
  pdl_wait();

  // ancestor-or-self mask of each row's node (its chain of parents)
  for (int rr = threadIdx.x; rr < ROWS; rr += blockDim.x) {
    const int r = row0 + rr;
    uint32_t* mw = mrow + (size_t)rr * a.W;
    for (int w = 0; w < a.W; ++w) mw[w] = 0u;
    if (r < nrows)
      for (int j = r / a.G; j >= 0; j = a.td.parent[j]) mw[j >> 5] |= 1u << (j & 31);
  }
  // queries of this CTA, pre-scaled so that exp2 gives the softmax weights
  for (int e = threadIdx.x; e < ROWS * DH; e += blockDim.x) {
    const int rr = e / DH, d = e - rr * DH;
    const int r = row0 + rr;
    float v = 0.f;
    if (r < nrows) {
      const int i = r / a.G, h = g * a.G + (r - i * a.G);
      v = to_f32(Q[(((size_t)b * a.T + i) * a.Hq + h) * DH + d]) * a.qscale;
    }
    qs[e] = v;
  }
  __syncthreads();

  float m[ROWS], l[ROWS], acc[ROWS][DPL];
#pragma unroll
  for (int rr = 0; rr < ROWS; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) acc[rr][t] = 0.f;
  }

  const int Lb = seq_len(a.lens, b, a.L, a.Lc, a.ws);
  const int n_cache_tiles = (Lb + KT - 1) / KT;
  const int n_tree_tiles = (a.T + KT - 1) / KT;
  const int key = lane % KT;  // the key this lane scores (lanes past KT repeat, their scores are dropped)
  for (int tile = warp; tile < n_cache_tiles + n_tree_tiles; tile += AF_WARPS) {
    const bool is_tree = tile >= n_cache_tiles;
    const int k0 = is_tree ? (tile - n_cache_tiles) * KT : tile * KT;
    const int nk = is_tree ? min(KT, a.T - k0) : min(KT, Lb - k0);
    __syncwarp();
    // the tile's K and V rows with 16-byte loads, a batch of AF_LB per lane
    // and array in flight before any is stored (keys past nk read as zero)
    {
      constexpr int VEC = 16 / (int)sizeof(TT);           // elements per 16-byte load
      constexpr int NV = KT * DH / VEC / 32;              // loads per lane and array
      constexpr int AF_LB = NV < 2 ? NV : 2;
      const TT* kb = reinterpret_cast<const TT*>(is_tree ? a.kt : a.kc);
      const TT* vb = reinterpret_cast<const TT*>(is_tree ? a.vt : a.vc);
      const int rows = is_tree ? a.T : a.Lc;
#pragma unroll
      for (int u0 = 0; u0 < NV; u0 += AF_LB) {
        uint4 kr[AF_LB], vr[AF_LB];
#pragma unroll
        for (int u = 0; u < AF_LB; ++u) {
          const int e = ((u0 + u) * 32 + lane) * VEC;  // element of the [KT][DH] tile
          const int j = e / DH, d = e - j * DH;
          kr[u] = make_uint4(0u, 0u, 0u, 0u);
          vr[u] = kr[u];
          if (j < nk) {
            const size_t o = (((size_t)b * rows + k0 + j) * a.Hkv + g) * DH + d;
            kr[u] = *reinterpret_cast<const uint4*>(kb + o);
            vr[u] = *reinterpret_cast<const uint4*>(vb + o);
          }
        }
#pragma unroll
        for (int u = 0; u < AF_LB; ++u) {
          const int e = ((u0 + u) * 32 + lane) * VEC;
          const int j = e / DH, d = e - j * DH;
          const TT* kx = reinterpret_cast<const TT*>(&kr[u]);
          const TT* vx = reinterpret_cast<const TT*>(&vr[u]);
#pragma unroll
          for (int x = 0; x < VEC; ++x) {
            ks[j * (DH + 1) + d + x] = to_f32(kx[x]);
            vs[j * DH + d + x] = to_f32(vx[x]);
          }
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
      const int r = row0 + rr;
      if (r >= nrows) break;
      float s = 0.f;
#pragma unroll 16
      for (int d = 0; d < DH; ++d) s = fmaf(qs[rr * DH + d], ks[key * (DH + 1) + d], s);
      bool ok = lane < KT && key < nk;
      if (is_tree) ok = ok && ((mrow[(size_t)rr * a.W + ((k0 + key) >> 5)] >> ((k0 + key) & 31)) & 1u);
      s = ok ? s : -INFINITY;
      const float mt = warp_max(s);
      if (mt == -INFINITY) continue;  // nothing visible in this tile
      const float mn = fmaxf(m[rr], mt);
      const float corr = exp2f(m[rr] - mn);  // 0 when m was -inf
      const float p = ok ? exp2f(s - mn) : 0.f;
      l[rr] = l[rr] * corr + warp_sum(p);
      m[rr] = mn;
#pragma unroll
      for (int t = 0; t < DPL; ++t) acc[rr][t] *= corr;
      for (int j = 0; j < nk; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int t = 0; t < DPL; ++t) acc[rr][t] = fmaf(pj, vs[j * DH + lane + 32 * t], acc[rr][t]);
      }
    }
  }

  // join the warps' states of every row: m* = max m_w,
  // o = sum_w 2^(m_w - m*) acc_w / sum_w 2^(m_w - m*) l_w
  __syncthreads();
  float* pm = qs + ROWS * DH;          // [AF_WARPS][ROWS] (reuses the tiles' space)
  float* pl = pm + AF_WARPS * ROWS;    // [AF_WARPS][ROWS]
  float* pa = pl + AF_WARPS * ROWS;    // [AF_WARPS][ROWS][DH]
#pragma unroll
  for (int rr = 0; rr < ROWS; ++rr) {
    if (lane == 0) {
      pm[warp * ROWS + rr] = m[rr];
      pl[warp * ROWS + rr] = l[rr];
    }
#pragma unroll
    for (int t = 0; t < DPL; ++t) pa[((size_t)warp * ROWS + rr) * DH + lane + 32 * t] = acc[rr][t];
  }
  __syncthreads();
  TT* O = reinterpret_cast<TT*>(a.out);
  for (int e = threadIdx.x; e < ROWS * DH; e += blockDim.x) {
    const int rr = e / DH, d = e - rr * DH;
    const int r = row0 + rr;
    if (r >= nrows) continue;
    float ms = -INFINITY;
    for (int w = 0; w < AF_WARPS; ++w) ms = fmaxf(ms, pm[w * ROWS + rr]);
    float num = 0.f, den = 0.f;
    for (int w = 0; w < AF_WARPS; ++w) {
      const float mw = pm[w * ROWS + rr];
      if (mw == -INFINITY) continue;  // this warp saw no visible key of the row
      const float f = exp2f(mw - ms);
      num = fmaf(f, pa[((size_t)w * ROWS + rr) * DH + d], num);
      den = fmaf(f, pl[w * ROWS + rr], den);
    }
    const int i = r / a.G, h = g * a.G + (r - i * a.G);
    O[((size_t)b * a.T + i) * a.H + (size_t)h * DH + d] = from_f32<TT>(num / den);
  }
}

// bf16, head dim 128: tcgen05 kernel (attn_tc.cu); other bf16: mma.sync kernel
// (attn_mma.cu); fp32: this CUDA-core kernel (no TF32)
int launch_tree_attn(const Plan& p, const void* q, const void* kt, const void* vt, const void* kc, const void* vc,
                     const int32_t* lens, void* out, uint8_t* ws, cudaStream_t st) {
  if (attn_tc_supported(p)) return launch_tree_attn_tc(p, q, kt, vt, kc, vc, lens, out, ws, st);
  if (p.bf16) return launch_tree_attn_mma(p, q, kt, vt, kc, vc, lens, out, ws, st);
  AttnArgs a;
  a.q = q;
  a.kt = kt;
  a.vt = vt;
  a.kc = kc;
  a.vc = vc;
  a.td = p.tree;
  a.out = out;
  a.B = p.B;
  a.T = p.T;
  a.W = p.W;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.G = p.G;
  a.L = p.L;
  a.Lc = p.Lc;
  a.H = p.H;
  a.qscale = 1.4426950408889634f / sqrtf((float)p.Dh);
  a.lens = lens;
  a.ws = ws;
  // 16 query rows per CTA; 2 when that leaves most SMs idle (a small tree
  // and batch): eight times the CTAs, each warp's row loop an eighth as long
  // (tiny-fp32: 30.7 -> 28.7 us per step, against 4 rows)
  const bool few = (long long)((p.T * p.G + AF_ROWS - 1) / AF_ROWS) * p.Hkv * p.B < 148;
  const int rows = few ? AF_ROWS_FEW : AF_ROWS;
  dim3 grid((p.T * p.G + rows - 1) / rows, p.Hkv, p.B);
  // the key tiles' space also holds the warps' final states ([8][rows] m and l, [8][rows][Dh] o)
  const size_t tiles = few ? (p.Dh == 128 ? af_smem_floats<128, AF_ROWS_FEW>() : af_smem_floats<64, AF_ROWS_FEW>())
                           : (p.Dh == 128 ? af_smem_floats<128, AF_ROWS>() : af_smem_floats<64, AF_ROWS>());
  const size_t join = (size_t)rows * p.Dh + 2 * AF_WARPS * rows + (size_t)AF_WARPS * rows * p.Dh;
  a.smem_floats = tiles > join ? tiles : join;
  const size_t smem = a.smem_floats * sizeof(float) + (size_t)rows * p.W * sizeof(uint32_t);
  void (*k)(AttnArgs);
  if (few) k = p.Dh == 128 ? tree_attn_kernel<float, 128, AF_ROWS_FEW> : tree_attn_kernel<float, 64, AF_ROWS_FEW>;
  else k = p.Dh == 128 ? tree_attn_kernel<float, 128, AF_ROWS> : tree_attn_kernel<float, 64, AF_ROWS>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_k(k, grid, dim3(AF_WARPS * 32), smem, st, true, a);
}

}  // namespace medusa
