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
// CUDA-core version: a CTA owns 32 query rows of one (b, g) and streams all
// of that group's keys through shared memory in tiles of 32 (cache tiles
// unmasked, tree tiles masked by one mask word per row and tile), with an
// fp32 online softmax per row in registers.  Rows of one (b, g) sit in
// adjacent CTAs so that the group's K/V tiles are served from L2 after the
// first read.  No split of the key range, so no partial results and no
// combine step.
#include "internal.cuh"

namespace medusa {

constexpr int AT_ROWS = 32;  // query rows per CTA (4 per warp)
constexpr int AT_KT = 32;    // keys per tile

struct AttnArgs {
  const void *q, *kt, *vt, *kc, *vc;
  const uint32_t* mask;  // [T][W]
  void* out;             // [B][T][H]
  int B, T, W, Hq, Hkv, G, L, Lc, H;
  float qscale;  // log2(e) / sqrt(Dh)
  const int32_t* lens;  // [B] per-sequence cache lengths, or null (L for all)
  uint8_t* ws;
};

template <typename TT, int DH>
__global__ void __launch_bounds__(256) tree_attn_kernel(AttnArgs a) {
  constexpr int DPL = DH / 32;  // dims per lane
  extern __shared__ float4 at_smem[];
  float(*qs)[DH] = reinterpret_cast<float(*)[DH]>(at_smem);                     // [AT_ROWS][DH]
  float(*ks)[DH + 1] = reinterpret_cast<float(*)[DH + 1]>(&qs[AT_ROWS][0]);     // [AT_KT][DH+1]
  float(*vs)[DH] = reinterpret_cast<float(*)[DH]>(&ks[AT_KT][0]);              // [AT_KT][DH]
  __shared__ uint32_t mw[AT_ROWS];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int row0 = blockIdx.x * AT_ROWS;
  const int nrows = a.T * a.G;
  const TT* Q = reinterpret_cast<const TT*>(a.q);
  pdl_trigger();
  pdl_wait();

  // queries of this CTA, pre-scaled so that exp2 gives the softmax weights
  for (int e = threadIdx.x; e < AT_ROWS * DH; e += blockDim.x) {
    const int rr = e / DH, d = e - rr * DH;
    const int r = row0 + rr;
    float v = 0.f;
    if (r < nrows) {
      const int i = r / a.G, h = g * a.G + (r - (r / a.G) * a.G);
      v = to_f32(Q[(((size_t)b * a.T + i) * a.Hq + h) * DH + d]) * a.qscale;
    }
    qs[rr][d] = v;
  }

  float m[4], l[4], acc[4][DPL];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) acc[rr][t] = 0.f;
  }

  const int Lb = seq_len(a.lens, b, a.L, a.Lc, a.ws);
  const int n_cache_tiles = (Lb + AT_KT - 1) / AT_KT;
  const int n_tree_tiles = (a.T + AT_KT - 1) / AT_KT;
  for (int tile = 0; tile < n_cache_tiles + n_tree_tiles; ++tile) {
    const bool is_tree = tile >= n_cache_tiles;
    const int k0 = is_tree ? (tile - n_cache_tiles) * AT_KT : tile * AT_KT;
    const int nk = is_tree ? min(AT_KT, a.T - k0) : min(AT_KT, Lb - k0);
    __syncthreads();
    for (int e = threadIdx.x; e < AT_KT * DH; e += blockDim.x) {
      const int j = e / DH, d = e - j * DH;
      float kv = 0.f, vv = 0.f;
      if (j < nk) {
        if (is_tree) {
          const size_t o = (((size_t)b * a.T + k0 + j) * a.Hkv + g) * DH + d;
          kv = to_f32(reinterpret_cast<const TT*>(a.kt)[o]);
          vv = to_f32(reinterpret_cast<const TT*>(a.vt)[o]);
        } else {
          const size_t o = (((size_t)b * a.Lc + k0 + j) * a.Hkv + g) * DH + d;
          kv = to_f32(reinterpret_cast<const TT*>(a.kc)[o]);
          vv = to_f32(reinterpret_cast<const TT*>(a.vc)[o]);
        }
      }
      ks[j][d] = kv;
      vs[j][d] = vv;
    }
    if (is_tree && threadIdx.x < AT_ROWS) {
      const int r = row0 + threadIdx.x;
      mw[threadIdx.x] = r < nrows ? a.mask[(size_t)(r / a.G) * a.W + (k0 >> 5)] : 0u;
    }
    __syncthreads();

#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int lr = warp * 4 + rr;
      if (row0 + lr >= nrows) continue;
      float s = 0.f;
#pragma unroll 16
      for (int d = 0; d < DH; ++d) s = fmaf(qs[lr][d], ks[lane][d], s);
      bool ok = lane < nk;
      if (is_tree) ok = ok && ((mw[lr] >> lane) & 1u);
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
        for (int t = 0; t < DPL; ++t) acc[rr][t] = fmaf(pj, vs[j][lane + 32 * t], acc[rr][t]);
      }
    }
  }

  TT* O = reinterpret_cast<TT*>(a.out);
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int r = row0 + warp * 4 + rr;
    if (r >= nrows) continue;
    const int i = r / a.G, h = g * a.G + (r - i * a.G);
    const float inv = 1.f / l[rr];
#pragma unroll
    for (int t = 0; t < DPL; ++t)
      O[((size_t)b * a.T + i) * a.H + (size_t)h * DH + lane + 32 * t] = from_f32<TT>(acc[rr][t] * inv);
  }
}

// bf16, head dim 128: tcgen05 kernel (attn_tc.cu); other bf16: mma.sync kernel
// (attn_mma.cu); fp32: this CUDA-core kernel (no TF32)
int launch_tree_attn(const Plan& p, const void* q, const void* kt, const void* vt, const void* kc, const void* vc,
                     const int32_t* lens, const uint32_t* mask, void* out, uint8_t* ws, cudaStream_t st) {
  if (attn_tc_supported(p)) return launch_tree_attn_tc(p, q, kt, vt, kc, vc, lens, out, ws, st);
  if (p.bf16) return launch_tree_attn_mma(p, q, kt, vt, kc, vc, lens, out, ws, st);
  AttnArgs a;
  a.q = q;
  a.kt = kt;
  a.vt = vt;
  a.kc = kc;
  a.vc = vc;
  a.mask = mask;
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
  dim3 grid((p.T * p.G + AT_ROWS - 1) / AT_ROWS, p.Hkv, p.B);
  const size_t smem = (size_t)(AT_ROWS * p.Dh + AT_KT * (p.Dh + 1) + AT_KT * p.Dh) * sizeof(float);
  void (*k)(AttnArgs);
  if (p.bf16) k = p.Dh == 128 ? tree_attn_kernel<__nv_bfloat16, 128> : tree_attn_kernel<__nv_bfloat16, 64>;
  else k = p.Dh == 128 ? tree_attn_kernel<float, 128> : tree_attn_kernel<float, 64>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_k(k, grid, dim3(256), smem, st, true, a);
}

}  // namespace medusa
