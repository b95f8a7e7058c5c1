// Tree attention with warp-level mma.sync (bf16, head dim 64), flash-style ("Medusa Heads",
// "Attenzione sull'albero e accettazione": all candidates in one pass, each
// seeing only its ancestors; "Tetes de decodage Medusa", "Plongee profonde").
//
//   o[b][i][h] = sum_j softmax_j(q . k_j / sqrt(Dh)) v_j
//   over cache rows j < L, then tree nodes j allowed by the node's mask row.
//
// A CTA owns 16*NW query rows (NW <= 12 warps: all rows of the (b, g) pair
// when they fit, so K/V are read once for all of them) of one (sequence b,
// kv head g); query row r is
// (node r / G, q head g*G + r % G).  Each warp holds 16 rows: their Q
// fragments stay in registers for the whole pass, S = Q K^T and O += P V are
// m16n8k16 bf16 MMAs with fp32 accumulation, the online softmax keeps its
// running max and sum per row in registers, and P is repacked from the S
// accumulators straight into A fragments.  K/V blocks of 64 keys stream
// through an S-deep cp.async ring in shared memory (rows padded to break
// bank conflicts); cache blocks need no mask, tree blocks test one mask bit per
// (row, key).  When (rows / 32) * Hkv * B is too small to fill the GPU the key
// range is split (flash-decoding): a few cache chunks plus one tree chunk per
// (b, g, row block), each writing an unnormalised partial (o, max, sum) that
// a small combine kernel merges; otherwise one CTA covers all keys and
// writes the output directly.
#include "internal.cuh"

namespace medusa {

constexpr int AM_KB = 64;  // keys per block

struct AmArgs {
  const __nv_bfloat16 *q, *kt, *vt, *kc, *vc;
  TreeDims td;  // the tree tables: each CTA derives its rows' ancestor masks from them
  __nv_bfloat16* out;
  int B, T, W, Hq, Hkv, G, L, Lc, H;
  int NS;          // key splits per (b, g): 1 = no split, else NS-1 cache chunks + the tree
  int chunk_blks;  // cache key blocks per cache chunk
  float* part_o;   // [B][Hq][T][NS][Dh] unnormalised partial outputs (split mode)
  float2* part_ml; // [B][Hq][T][NS] (running max in log2 units, sum)
  float qscale;    // log2(e) / sqrt(Dh)
  const int32_t* lens;  // [B] per-sequence cache lengths, or null (L for all)
  uint8_t* ws;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int DH, int NW, int S>
__global__ void __launch_bounds__(NW * 32, 1) tree_attn_mma_kernel(const __grid_constant__ AmArgs a) {
  constexpr int LD = DH + 8;  // padded smem row (elements)
  constexpr int NT = NW * 32;
  constexpr int KS = DH / 16;  // k-steps of Q K^T
  constexpr int ND = DH / 8;   // n-tiles of O
  extern __shared__ float4 am_smem[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(am_smem);  // [S][AM_KB][LD]
  __nv_bfloat16* Vs = Ks + S * AM_KB * LD;                          // [S][AM_KB][LD]
  uint32_t* mrow = reinterpret_cast<uint32_t*>(Vs + S * AM_KB * LD);  // [16*NW][W] ancestor-or-self bits

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;  // mma group / thread-in-group
  const int g = blockIdx.y / a.NS, sp = blockIdx.y - g * a.NS, b = blockIdx.z;
  const int nrows = a.T * a.G;
  const int rbase = blockIdx.x * 16 * NW + warp * 16;
  const size_t kv_row = (size_t)a.Hkv * DH;  // elements between consecutive keys
  pdl_trigger();
  // Ancestor-or-self mask rows of this CTA's query rows (chains of parents).
  // The kernel reads nothing an earlier kernel of the step writes.
  for (int rr = threadIdx.x; rr < 16 * NW; rr += NT) {
    const int r = blockIdx.x * 16 * NW + rr;
    uint32_t* mr = mrow + (size_t)rr * a.W;
    for (int w = 0; w < a.W; ++w) mr[w] = 0u;
    if (r < nrows)
      for (int j = r / a.G; j >= 0; j = a.td.parent[j]) mr[j >> 5] |= 1u << (j & 31);
  }
  __syncthreads();

  // ---- Q fragments (rows gq and gq+8 of this warp), scale folded in later
  uint32_t qf[KS][4];
  int node[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = rbase + gq + hr * 8;
    const bool ok = r < nrows;
    const int i = ok ? r / a.G : 0;
    node[hr] = ok ? i : -1;
    const int h = g * a.G + (ok ? r - i * a.G : 0);
    const __nv_bfloat16* qp = a.q + (((size_t)b * a.T + i) * a.Hq + h) * DH;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const uint32_t lo = ok ? *reinterpret_cast<const uint32_t*>(qp + kk * 16 + 2 * tq) : 0u;
      const uint32_t hi = ok ? *reinterpret_cast<const uint32_t*>(qp + kk * 16 + 8 + 2 * tq) : 0u;
      qf[kk][hr] = lo;       // a0 (row gq) / a1 (row gq+8)
      qf[kk][hr + 2] = hi;   // a2 / a3
    }
  }

  float o[ND][4];
#pragma unroll
  for (int j = 0; j < ND; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow_m[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const int Lb = seq_len(a.lens, b, a.L, a.Lc, a.ws);
  const int nb_cache = (Lb + AM_KB - 1) / AM_KB;
  const int nb_tree = (a.T + AM_KB - 1) / AM_KB;
  // this CTA's key blocks [blk_lo, blk_hi) of (cache blocks, then tree blocks)
  // split sp takes an equal share of the concatenated (cache, tree) block list
  const int nb_all = nb_cache + nb_tree;
  const int blk_lo = (int)(((long long)sp * nb_all) / a.NS);
  const int blk_hi = (int)(((long long)(sp + 1) * nb_all) / a.NS);

  auto load_block = [&](int blk, int buf) {
    const bool tree = blk >= nb_cache;
    const int k0 = tree ? (blk - nb_cache) * AM_KB : blk * AM_KB;
    const int nk = tree ? min(AM_KB, a.T - k0) : min(AM_KB, Lb - k0);
    const __nv_bfloat16* kb = tree ? a.kt + ((size_t)b * a.T) * kv_row : a.kc + ((size_t)b * a.Lc) * kv_row;
    const __nv_bfloat16* vb = tree ? a.vt + ((size_t)b * a.T) * kv_row : a.vc + ((size_t)b * a.Lc) * kv_row;
    constexpr int CH = DH / 8;  // 16-byte chunks per row
    for (int c = threadIdx.x; c < AM_KB * CH; c += NT) {
      const int j = c / CH, x = (c - j * CH) * 8;
      const bool ok = j < nk;
      const size_t src = ((size_t)(ok ? k0 + j : k0)) * kv_row + (size_t)g * DH + x;
      cp_async16(Ks + ((size_t)buf * AM_KB + j) * LD + x, kb + src, ok);
      cp_async16(Vs + ((size_t)buf * AM_KB + j) * LD + x, vb + src, ok);
    }
    cp_async_commit();
  };

  // S-deep ring: S-1 blocks in flight ahead of the one being computed (one
  // cp.async group per block; empty groups keep the count uniform)
#pragma unroll
  for (int pi = 0; pi < S - 1; ++pi) {
    if (blk_lo + pi < blk_hi) load_block(blk_lo + pi, pi);
    else cp_async_commit();
  }
  for (int blk = blk_lo; blk < blk_hi; ++blk) {
    const int i = blk - blk_lo;
    const int buf = i % S;
    if (blk + S - 1 < blk_hi) load_block(blk + S - 1, (i + S - 1) % S);
    else cp_async_commit();
    cp_async_wait<S - 1>();  // every group but the S-1 newest has landed: block blk is in
    __syncthreads();

    const bool tree = blk >= nb_cache;
    const int k0 = tree ? (blk - nb_cache) * AM_KB : blk * AM_KB;
    const int nk = tree ? min(AM_KB, a.T - k0) : min(AM_KB, Lb - k0);
    const __nv_bfloat16* Kb = Ks + (size_t)buf * AM_KB * LD;
    const __nv_bfloat16* Vb = Vs + (size_t)buf * AM_KB * LD;
    if (rbase >= nrows) {  // all 16 rows of this warp are padding: no math, keep the barriers
      __syncthreads();
      continue;
    }

    // ---- S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int kk = 0; kk < KS; kk += 2) {
        uint32_t bf[4];  // b0,b1 of k-step kk and kk+1
        const int mi = lane >> 3, ri = lane & 7;
        ldsm_x4(bf, Kb + (size_t)(nt * 8 + ri) * LD + kk * 16 + mi * 8);
        mma16816(s[nt], qf[kk], bf[0], bf[1]);
        mma16816(s[nt], qf[kk + 1], bf[2], bf[3]);
      }
    }
    // ---- mask, scale, online softmax (rows gq and gq+8)
    uint32_t mw[2][2] = {{0u, 0u}, {0u, 0u}};
    if (tree) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
        if (node[hr] >= 0) {
          const int w0 = k0 >> 5;
          const uint32_t* mr = mrow + (size_t)(warp * 16 + gq + hr * 8) * a.W;
          mw[hr][0] = mr[w0];
          mw[hr][1] = (w0 + 1 < a.W) ? mr[w0 + 1] : 0u;
        }
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        const int kl = nt * 8 + 2 * tq + (e & 1);  // key within the block
        bool ok = kl < nk;
        if (tree) ok = ok && ((mw[hr][kl >> 5] >> (kl & 31)) & 1u);
        const float v = ok ? s[nt][e] * a.qscale : -INFINITY;
        s[nt][e] = v;
        mx[hr] = fmaxf(mx[hr], v);
      }
    float corr[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      const float mn = fmaxf(mrow_m[hr], mx[hr]);
      // mn == -inf: nothing visible yet for this row; keep everything at zero
      corr[hr] = (mn == -INFINITY) ? 1.f : exp2f(mrow_m[hr] - mn);
      mrow_m[hr] = mn;
    }
    float ls[2] = {0.f, 0.f};
    uint32_t pf[4][4];  // A fragments of P for the 4 k-steps of P V
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        p[e] = (s[nt][e] == -INFINITY) ? 0.f : exp2f(s[nt][e] - mrow_m[hr]);
        ls[hr] += p[e];
      }
      const int kk2 = nt >> 1, half = nt & 1;
      pf[kk2][half * 2 + 0] = pack_bf16(p[0], p[1]);  // row gq
      pf[kk2][half * 2 + 1] = pack_bf16(p[2], p[3]);  // row gq+8
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      ls[hr] += __shfl_xor_sync(0xffffffffu, ls[hr], 1);
      ls[hr] += __shfl_xor_sync(0xffffffffu, ls[hr], 2);
      lrow[hr] = lrow[hr] * corr[hr] + ls[hr];
    }
#pragma unroll
    for (int j = 0; j < ND; ++j) {
      o[j][0] *= corr[0];
      o[j][1] *= corr[0];
      o[j][2] *= corr[1];
      o[j][3] *= corr[1];
    }
    // ---- O += P V: 4 k-steps of 16 keys, ND n-tiles of 8 dims
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
      // A fragment order: a0 (row gq, keys 0-7 of the step), a1 (row gq+8, 0-7), a2 (row gq, 8-15), a3 (gq+8, 8-15)
      const uint32_t af[4] = {pf[kk2][0], pf[kk2][1], pf[kk2][2], pf[kk2][3]};
#pragma unroll
      for (int j = 0; j < ND; j += 2) {
        uint32_t bf[4];  // (keys 0-7, dims j), (keys 8-15, dims j), (keys 0-7, dims j+1), (keys 8-15, dims j+1)
        const int mi = lane >> 3, ri = lane & 7;
        const int key = kk2 * 16 + (mi & 1) * 8 + ri;
        const int dim = (j + (mi >> 1)) * 8;
        ldsm_x4_t(bf, Vb + (size_t)key * LD + dim);
        mma16816(o[j], af, bf[0], bf[1]);
        mma16816(o[j + 1], af, bf[2], bf[3]);
      }
    }
    __syncthreads();  // this buffer is refilled S-1 blocks later
  }

  // ---- split mode: unnormalised partial; else normalise and store (bf16)
  if (a.NS > 1) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = rbase + gq + hr * 8;
      if (r >= nrows) continue;
      const int i = r / a.G, h = g * a.G + (r - (r / a.G) * a.G);
      const size_t pr = (((size_t)b * a.Hq + h) * a.T + i) * a.NS + sp;
      float* po = a.part_o + pr * DH;
#pragma unroll
      for (int j = 0; j < ND; ++j)
        *reinterpret_cast<float2*>(po + j * 8 + 2 * tq) = make_float2(o[j][hr * 2], o[j][hr * 2 + 1]);
      if (tq == 0) a.part_ml[pr] = make_float2(mrow_m[hr], lrow[hr]);
    }
    pdl_wait();  // completes only after the preceding kernel (keeps the stream's order transitive)
    return;
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = rbase + gq + hr * 8;
    if (r >= nrows) continue;
    const int i = r / a.G, h = g * a.G + (r - (r / a.G) * a.G);
    const float inv = 1.f / lrow[hr];
    __nv_bfloat16* op = a.out + ((size_t)b * a.T + i) * a.H + (size_t)h * DH;
#pragma unroll
    for (int j = 0; j < ND; ++j)
      *reinterpret_cast<uint32_t*>(op + j * 8 + 2 * tq) = pack_bf16(o[j][hr * 2] * inv, o[j][hr * 2 + 1] * inv);
  }
  pdl_wait();  // completes only after the preceding kernel (keeps the stream's order transitive)
}

// Merges the NS partials of every (b, q head, node): one warp per row.
template <int DH>
__global__ void __launch_bounds__(256) tree_attn_combine_kernel(const __grid_constant__ AmArgs a) {
  const int lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // (b, h, i) flattened
  pdl_trigger();
  pdl_wait();
  if (row >= (size_t)a.B * a.Hq * a.T) return;
  const int i = (int)(row % a.T);
  const int h = (int)((row / a.T) % a.Hq);
  const int b = (int)(row / ((size_t)a.T * a.Hq));
  float mx = -INFINITY;
  for (int s = 0; s < a.NS; ++s) mx = fmaxf(mx, a.part_ml[row * a.NS + s].x);
  float acc[DH / 32], l = 0.f;
#pragma unroll
  for (int t = 0; t < DH / 32; ++t) acc[t] = 0.f;
  for (int s = 0; s < a.NS; ++s) {
    const float2 ml = a.part_ml[row * a.NS + s];
    if (ml.x == -INFINITY) continue;  // a split that saw no key (its partial output is not read)
    const float w = exp2f(ml.x - mx);
    l += w * ml.y;
    const float* po = a.part_o + (row * a.NS + s) * DH;
#pragma unroll
    for (int t = 0; t < DH / 32; ++t) acc[t] += w * po[lane + 32 * t];
  }
  const float inv = 1.f / l;
  __nv_bfloat16* op = a.out + ((size_t)b * a.T + i) * a.H + (size_t)h * DH;
#pragma unroll
  for (int t = 0; t < DH / 32; ++t) op[lane + 32 * t] = __float2bfloat16_rn(acc[t] * inv);
}

// Key splits for a shape (device independent, so the workspace can be sized
// from the config alone): split when fewer than ~2 waves of 2-warp CTAs exist.
// Warps per CTA (16 query rows each) for a shape: all rows of one (b, kv head)
// in one CTA when they fit 12 warps (K/V blocks are then loaded once for every
// row), else row blocks of 12 warps.
static int attn_warps(int rows) {
  if (rows <= 64) return 4;
  if (rows <= 128) return 8;
  return 12;
}

// Key splits for a shape (device independent, so the workspace can be sized
// from the config alone): when the (row block, b, kv head) CTAs do not cover
// the ~148 SMs of a B300, the key blocks (cache blocks, then tree blocks) are
// cut into NS equal shares, each CTA writing a partial that the combine
// kernel merges.
void attn_split_shape(int B, int T, int G, int Hkv, int L, int* NS, int* chunk_blks) {
  constexpr int kSlots = 148;
  const int rows = T * G;
  const int nw = attn_warps(rows);
  const int row_blocks = (rows + 16 * nw - 1) / (16 * nw);
  const int base = row_blocks * Hkv * B;
  const int nb_all = (L + AM_KB - 1) / AM_KB + (T + AM_KB - 1) / AM_KB;
  *NS = 1;
  *chunk_blks = nb_all;
  if (2 * base > kSlots || L == 0) return;
  int ns = kSlots / base;
  if (ns > nb_all) ns = nb_all;
  if (ns < 2) return;
  *NS = ns;
  *chunk_blks = (nb_all + ns - 1) / ns;
}

// sized for the larger key split of the two bf16 attention kernels
size_t attn_part_bytes(int B, int T, int G, int Hkv, int L, int Dh) {
  int NS, cb;
  attn_split_shape(B, T, G, Hkv, L, &NS, &cb);
  if (Dh == 128) {
    const int ns_tc = attn_tc_splits(B, T, G, Hkv, L);
    if (ns_tc > NS) NS = ns_tc;
  }
  if (NS == 1) return 0;
  const size_t rows = (size_t)B * Hkv * G * T * NS;
  return rows * Dh * sizeof(float) + rows * sizeof(float2) + 256;
}

int launch_tree_attn_mma(const Plan& p, const void* q, const void* kt, const void* vt, const void* kc, const void* vc,
                         const int32_t* lens, void* out, uint8_t* ws, cudaStream_t st) {
  AmArgs a;
  a.q = (const __nv_bfloat16*)q;
  a.kt = (const __nv_bfloat16*)kt;
  a.vt = (const __nv_bfloat16*)vt;
  a.kc = (const __nv_bfloat16*)(kc ? kc : kt);
  a.vc = (const __nv_bfloat16*)(vc ? vc : vt);
  a.td = p.tree;
  a.out = (__nv_bfloat16*)out;
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
  attn_split_shape(p.B, p.T, p.G, p.Hkv, p.L, &a.NS, &a.chunk_blks);
  const size_t rows_all = (size_t)p.B * p.Hq * p.T * a.NS;
  a.part_o = reinterpret_cast<float*>(ws + p.off_attn_part);
  a.part_ml = reinterpret_cast<float2*>(ws + p.off_attn_part + rows_all * p.Dh * sizeof(float));
  const int rows = p.T * p.G;
  const int nw = attn_warps(rows);
  dim3 grid((rows + 16 * nw - 1) / (16 * nw), p.Hkv * a.NS, p.B);
  // a 4-block ring (one CTA per SM) when the grid is a single wave, else a
  // 2-block ring so that several CTAs share an SM
  const int ctas = (int)(grid.x * grid.y * grid.z);
  const int S = ctas <= p.sm_count ? 4 : 2;
  const size_t smem = (size_t)2 * S * AM_KB * (p.Dh + 8) * sizeof(__nv_bfloat16) +
                      (size_t)16 * nw * p.W * sizeof(uint32_t);
  void (*k)(AmArgs) = nullptr;
#define AM_PICK(D, W, SS) \
  if (p.Dh == D && nw == W && S == SS) k = tree_attn_mma_kernel<D, W, SS>;
  // head dim 128 runs on the tensor-core kernel (attn_tc.cu)
  AM_PICK(64, 4, 2) AM_PICK(64, 8, 2) AM_PICK(64, 12, 2) AM_PICK(64, 4, 4) AM_PICK(64, 8, 4) AM_PICK(64, 12, 4)
#undef AM_PICK
  if (!k) return (int)cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return (int)e;
  e = launch_k(k, grid, dim3(nw * 32), smem, st, false, a);
  if (e != cudaSuccess || a.NS == 1) return (int)e;
  const size_t nrow = (size_t)p.B * p.Hq * p.T;
  const unsigned cgrid = (unsigned)((nrow + 7) / 8);
  if (p.Dh == 128) return (int)launch_k(tree_attn_combine_kernel<128>, dim3(cgrid), dim3(256), 0, st, true, a);
  return (int)launch_k(tree_attn_combine_kernel<64>, dim3(cgrid), dim3(256), 0, st, true, a);
}

// Merge of NS key-split partials ([B][Hq][T][NS] rows of Dh fp32 plus
// (max, sum)) written by either attention kernel.
int launch_attn_combine(const Plan& p, float* part_o, float2* part_ml, int NS, void* out, cudaStream_t st) {
  AmArgs a{};
  a.out = (__nv_bfloat16*)out;
  a.B = p.B;
  a.T = p.T;
  a.Hq = p.Hq;
  a.H = p.H;
  a.NS = NS;
  a.part_o = part_o;
  a.part_ml = part_ml;
  const size_t nrow = (size_t)p.B * p.Hq * p.T;
  const unsigned cgrid = (unsigned)((nrow + 7) / 8);
  if (p.Dh == 128) return (int)launch_k(tree_attn_combine_kernel<128>, dim3(cgrid), dim3(256), 0, st, true, a);
  return (int)launch_k(tree_attn_combine_kernel<64>, dim3(cgrid), dim3(256), 0, st, true, a);
}

}  // namespace medusa
