// Cartesian candidate tree ("Medusa Heads", "Attenzione sull'albero e
// accettazione": the heads' best tokens combined by Cartesian product into a
// prefix-sharing tree; each token may attend only to its own ancestors).
//
// Layout (closed form, no search): level d holds prod_{j<=d} k_j nodes
// starting at off[d]; the node with local index m at level d has rank
// m % k_d in the head-d list and parent off[d-1] + m / k_d (the root for
// d = 1).  One thread per (sequence, node) fills the tokens; the
// sequence-independent arrays (parent, depth, rank, pos, mask rows, leaf
// paths) are written by the first threads.
#include "internal.cuh"

namespace medusa {

struct TreeArgs {
  TreeDims td;
  int B, K, kmax, L;
  const int32_t* topk_idx;  // [B][K][kmax]
  const int32_t* root;      // [B]
  medusa_tree_t t;
};

__device__ __forceinline__ int node_depth(const TreeDims& td, int i) {
  int d = 0;
#pragma unroll 1
  for (int e = 1; e <= td.D; ++e)
    if (i >= td.off[e]) d = e;
  return d;
}

__device__ __forceinline__ int node_parent(const TreeDims& td, int i, int d) {
  if (d == 0) return -1;
  const int m = i - td.off[d];
  return d == 1 ? 0 : td.off[d - 1] + m / td.k[d];
}

__global__ void tree_build_kernel(TreeArgs a) {
  const TreeDims& td = a.td;
  const int gid = blockIdx.x * blockDim.x + threadIdx.x;
  const int T = td.T;
  pdl_trigger();
  if (gid < a.B * T) {
    pdl_wait();  // the top-k lists come from the previous kernel
    const int b = gid / T, i = gid - b * T;
    const int d = node_depth(td, i);
    int tok;
    if (d == 0) {
      tok = a.root[b];
    } else {
      const int rank = (i - td.off[d]) % td.k[d];
      tok = a.topk_idx[((size_t)b * a.K + (d - 1)) * a.kmax + rank];
    }
    a.t.token[(size_t)b * T + i] = tok;
  }
  if (gid < T) {
    const int i = gid;
    const int d = node_depth(td, i);
    a.t.depth[i] = d;
    a.t.parent[i] = node_parent(td, i, d);
    a.t.rank[i] = d == 0 ? 0 : (i - td.off[d]) % td.k[d];
    a.t.pos[i] = a.L + d;
    // mask row: one 32-bit word at a time, setting the bits of the chain to the root
    for (int w = 0; w < td.W; ++w) {
      uint32_t word = 0;
      int j = i, dj = d;
      while (j >= 0) {
        if ((j >> 5) == w) word |= 1u << (j & 31);
        const int pj = node_parent(td, j, dj);
        j = pj;
        dj -= 1;
      }
      a.t.mask[(size_t)i * td.W + w] = word;
    }
  }
  if (gid < td.n_leaves) {
    int j = td.off[td.D] + gid;
    for (int d = td.D; d >= 0; --d) {
      a.t.paths[(size_t)gid * (td.D + 1) + d] = j;
      j = node_parent(td, j, d);
    }
  }
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
