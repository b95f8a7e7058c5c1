// Candidate tree ("Medusa Heads", "Attenzione sull'albero e accettazione":
// the heads' best tokens combined into a prefix-sharing tree -- the Cartesian
// product of the lists, or a caller's subset of it; each token may attend only
// to its own ancestors).
//
// The layout tables (parent, depth, rank, children, leaves) come from the
// host plan; a node's token is the rank-th entry of the head list of its
// depth.  One thread per (sequence, node) fills the tokens; the sequence-
// independent arrays (parent, depth, rank, pos, mask rows, leaf paths) are
// written by the first threads.
#include "internal.cuh"

namespace medusa {

struct TreeArgs {
  TreeDims td;
  int B, K, kmax, L;
  const int32_t* topk_idx;  // [B][K][kmax]
  const int32_t* root;      // [B]
  medusa_tree_t t;
};

// mask row word w of node i: the bits of the nodes on its chain to the root
__device__ __forceinline__ uint32_t mask_word(const TreeDims& td, int i, int w) {
  uint32_t word = 0;
  for (int j = i; j >= 0; j = td.parent[j])
    if ((j >> 5) == w) word |= 1u << (j & 31);
  return word;
}

// the sequence-independent tree arrays, node i / leaf l
__device__ __forceinline__ void write_node(const TreeDims& td, const medusa_tree_t& t, int L, int i) {
  t.depth[i] = td.depth[i];
  t.parent[i] = td.parent[i];
  t.rank[i] = td.rank[i];
  t.pos[i] = L + td.depth[i];
  for (int w = 0; w < td.W; ++w) t.mask[(size_t)i * td.W + w] = mask_word(td, i, w);
}
__device__ __forceinline__ void write_path(const TreeDims& td, const medusa_tree_t& t, int l) {
  const int leaf = td.leaf[l], dl = td.depth[leaf];
  for (int d = td.D; d > dl; --d) t.paths[(size_t)l * (td.D + 1) + d] = -1;
  int j = leaf;
  for (int d = dl; d >= 0; --d) {
    t.paths[(size_t)l * (td.D + 1) + d] = j;
    j = td.parent[j];
  }
}

__global__ void tree_build_kernel(const __grid_constant__ TreeArgs a) {
  const TreeDims& td = a.td;
  const int gid = blockIdx.x * blockDim.x + threadIdx.x;
  const int T = td.T;
  pdl_trigger();
  pdl_wait();  // the top-k lists come from the previous kernel, which may also still read the tree
  if (gid < a.B * T && a.topk_idx) {  // (no lists: the sequence-independent arrays only)
    const int b = gid / T, i = gid - b * T;
    const int d = td.depth[i];
    const int tok = d == 0 ? a.root[b] : a.topk_idx[((size_t)b * a.K + (d - 1)) * a.kmax + td.rank[i]];
    a.t.token[(size_t)b * T + i] = tok;
  }
  if (gid < T) write_node(td, a.t, a.L, gid);
  if (gid < td.n_leaves) write_path(td, a.t, gid);
}

// ---------------------------------------------------------------------------
// Fused step: final per-head top-k merge and the tree in one kernel, one CTA
// per sequence.  Warp k merges head k's per-CTA candidate lists (written by
// the projection kernel: cand[cta][piece][sequence][kmax], the piece's head
// in cand_seg[cta][piece]); every slot's loads are issued before any is
// used.  The merged lists go to the topk outputs and to shared memory, from
// which the same CTA fills the sequence's tree tokens; CTA 0 also writes the
// sequence-independent arrays.
struct MergeTreeArgs {
  TreeArgs t;
  int S, rpc, nctas;  // work units per head, units per projection CTA (CTA c has [c*rpc, (c+1)*rpc)), CTAs
  int topk_n[MEDUSA_MAX_HEADS];
  const float* cand_val;
  const int* cand_idx;
  const int* cand_seg;
  int32_t* out_idx;  // [B][K][kmax]
  float* out_val;
  // The projection's CTAs each raise this count once their candidates are
  // written.  With it the kernel runs beside the verification projection (its
  // preceding grid, which reads nothing of this kernel's): it waits for the
  // count instead of that grid, and waits for the grid only at its end, so
  // that its completion still implies the completion of everything before it.
  const int* proj_done;
  uint8_t* ws;
};

__device__ __forceinline__ bool mt_better(float v, int i, float w, int j) { return v > w || (v == w && i < j); }

template <int KM>
__global__ void __launch_bounds__(256) merge_tree_kernel(const __grid_constant__ MergeTreeArgs a) {
  __shared__ int s_idx[MEDUSA_MAX_HEADS][MEDUSA_MAX_TOPK];
  __shared__ int16_t s_parent[MEDUSA_MAX_NODES];
  __shared__ uint8_t s_depth[MEDUSA_MAX_NODES], s_rank[MEDUSA_MAX_NODES];
  const TreeArgs& ta = a.t;
  const TreeDims& td = ta.td;
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  // the tree tables move to shared memory first: the walks below index them
  // with data-dependent node ids, which parameter space serves slowly
  for (int i = threadIdx.x; i < td.T; i += blockDim.x) {
    s_parent[i] = td.parent[i];
    s_depth[i] = td.depth[i];
    s_rank[i] = td.rank[i];
  }
  if (a.proj_done) {  // the candidates: every projection CTA has counted itself
    if (threadIdx.x == 0) wait_count(a.proj_done, a.nctas, 20ull * 1000 * 1000, a.ws);
  } else {
    pdl_wait();  // the candidates come from the preceding grid, the projection
  }
  __syncthreads();
  if (warp < ta.K) {
    const int seg = warp;
    int kn = 1;
#pragma unroll
    for (int k = 0; k < MEDUSA_MAX_HEADS; ++k)
      if (k == seg) kn = a.topk_n[k];
    const int b_lo = (int)(((long long)seg * a.S) / a.rpc);
    const int b_hi = min(a.nctas - 1, (int)(((long long)(seg + 1) * a.S - 1) / a.rpc));
    const int n_slots = (b_hi - b_lo + 1) * kMaxPieces;
    float lv[KM];
    int li[KM];
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      lv[i] = -INFINITY;
      li[i] = INT_MAX;
    }
    for (int sl0 = 0; sl0 < n_slots; sl0 += 32 * 4) {
      int sg[4];
      float cv[4][KM];
      int ci[4][KM];
#pragma unroll
      for (int u = 0; u < 4; ++u) {  // all loads of this round first
        const int sl = sl0 + u * 32 + lane;
        const bool in = sl < n_slots;
        const int blk = b_lo + sl / kMaxPieces, pc = sl % kMaxPieces;
        sg[u] = in ? __ldcg(a.cand_seg + blk * kMaxPieces + pc) : -1;
        const size_t base = ((size_t)(blk * kMaxPieces + pc) * ta.B + b) * ta.kmax;
#pragma unroll
        for (int i = 0; i < KM; ++i) {
          const bool ok = in && i < kn;
          cv[u][i] = ok ? __ldcg(a.cand_val + base + i) : -INFINITY;
          ci[u][i] = ok ? __ldcg(a.cand_idx + base + i) : INT_MAX;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (sg[u] != seg) continue;
#pragma unroll
        for (int i = 0; i < KM; ++i) {  // compare-and-swap insertion of candidate i
          float v = cv[u][i];
          int id = ci[u][i];
#pragma unroll
          for (int j = 0; j < KM; ++j) {
            const bool sw = (j < kn) && mt_better(v, id, lv[j], li[j]);
            const float ov = lv[j];
            const int oi = li[j];
            lv[j] = sw ? v : ov;
            li[j] = sw ? id : oi;
            v = sw ? ov : v;
            id = sw ? oi : id;
          }
        }
      }
    }
    // warp-wide top-kn: the best list head wins each round, its owner pops
    for (int rnk = 0; rnk < ta.kmax; ++rnk) {
      float bv = lv[0];
      int bi = li[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (mt_better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi != INT_MAX && lv[0] == bv && li[0] == bi) {
#pragma unroll
        for (int i = 0; i < KM - 1; ++i) {
          lv[i] = lv[i + 1];
          li[i] = li[i + 1];
        }
        lv[KM - 1] = -INFINITY;
        li[KM - 1] = INT_MAX;
      }
      if (lane == 0) {
        const bool live = rnk < kn && bi != INT_MAX;
        const size_t o = ((size_t)b * ta.K + seg) * ta.kmax + rnk;
        a.out_idx[o] = live ? bi : -1;
        a.out_val[o] = live ? bv : -INFINITY;
        s_idx[seg][rnk] = live ? bi : -1;
      }
    }
  }
  __syncthreads();
  const int T = td.T, W = td.W;
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    const int d = s_depth[i];
    ta.t.token[(size_t)b * T + i] = d == 0 ? ta.root[b] : s_idx[d - 1][s_rank[i]];
    if (b == 0) {
      ta.t.depth[i] = d;
      ta.t.parent[i] = s_parent[i];
      ta.t.rank[i] = s_rank[i];
      ta.t.pos[i] = ta.L + d;
    }
  }
  if (b == 0) {
    for (int e = threadIdx.x; e < T * W; e += blockDim.x) {  // mask word w of node i
      const int i = e / W, w = e - i * W;
      uint32_t word = 0;
      for (int j = i; j >= 0; j = s_parent[j])
        if ((j >> 5) == w) word |= 1u << (j & 31);
      ta.t.mask[e] = word;
    }
    for (int l = threadIdx.x; l < td.n_leaves; l += blockDim.x) {  // root-to-leaf path, then -1
      const int leaf = td.leaf[l], dl = s_depth[leaf];
      int32_t* row = ta.t.paths + (size_t)l * (td.D + 1);
      for (int d = td.D; d > dl; --d) row[d] = -1;
      for (int d = dl, j = leaf; d >= 0; --d, j = s_parent[j]) row[d] = j;
    }
  }
  if (a.proj_done) pdl_wait();  // complete only after the preceding grid
}

int launch_merge_tree(const Plan& p, int32_t* topk_idx, float* topk_val, const int32_t* root,
                      const medusa_tree_t& t, uint8_t* ws, int nctas, int rpc, int S, bool count_wait,
                      cudaStream_t st) {
  MergeTreeArgs a;
  a.t.td = p.tree;
  a.t.B = p.B;
  a.t.K = p.K;
  a.t.kmax = p.kmax;
  a.t.L = p.L;
  a.t.topk_idx = topk_idx;
  a.t.root = root;
  a.t.t = t;
  a.S = S;
  a.rpc = rpc;
  a.nctas = nctas;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.topk_n[k] = p.topk_n[k];
  a.cand_val = reinterpret_cast<const float*>(ws + p.off_cand_val);
  a.cand_idx = reinterpret_cast<const int*>(ws + p.off_cand_idx);
  a.cand_seg = reinterpret_cast<const int*>(ws + p.off_cand_seg);
  a.out_idx = topk_idx;
  a.out_val = topk_val;
  a.proj_done = count_wait ? reinterpret_cast<const int*>(ws) + TICKET_PROJ_DONE : nullptr;
  a.ws = ws;
  if (p.kmax <= 4) return (int)launch_k(merge_tree_kernel<4>, dim3(p.B), dim3(256), 0, st, true, a);
  if (p.kmax <= 8) return (int)launch_k(merge_tree_kernel<8>, dim3(p.B), dim3(256), 0, st, true, a);
  return (int)launch_k(merge_tree_kernel<MEDUSA_MAX_TOPK>, dim3(p.B), dim3(256), 0, st, true, a);
}

int launch_tree_build(const Plan& p, const int32_t* topk_idx, const int32_t* root, const medusa_tree_t& t,
                      cudaStream_t st) {
  TreeArgs a;
  a.td = p.tree;
  a.B = p.B;
  a.K = p.K;
  a.kmax = p.kmax;
  a.L = p.L;
  a.topk_idx = topk_idx;
  a.root = root;
  a.t = t;
  int n = p.B * p.T;
  if (p.T > n) n = p.T;
  if (p.NL > n) n = p.NL;
  const int threads = 256;
  return (int)launch_k(tree_build_kernel, dim3((n + threads - 1) / threads), dim3(threads), 0, st, true, a);
}

}  // namespace medusa
