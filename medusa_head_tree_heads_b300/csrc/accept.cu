// Acceptance ("Medusa Heads", "Attenzione sull'albero e accettazione": with
// greedy decoding a candidate is accepted when it equals the model's top
// choice; typical acceptance keeps a candidate whose base-model probability
// exceeds a threshold tied to the entropy of the distribution; the longest
// accepted branch is kept.  "Tetes de decodage Medusa", "Plongee profonde":
// the longest prefix matching what the model would have produced).
//
// One CTA per sequence.  Every non-root node c defines the edge
// parent(c) -> c; its keep flag is computed in parallel (typical mode scores
// token_c under the parent's distribution with one dot product
// lm_head[token_c] . o_parent: for bf16 the verification merge has already
// done so, one warp per parent), then every leaf path counts its leading kept
// edges and a block reduction picks the longest (ties: the smaller last kept
// node, which in breadth-first (depth, parent, rank) order is the lower node at
// the first divergence).
#include <limits.h>

#include "internal.cuh"

namespace medusa {


struct AcceptArgs {
  int B, T, D, NL, V, H;
  int typical;
  float inv_temp, log_eps, log_delta;
  const void* attn_out;  // [B][T][H]
  const void* lm_head;   // [V][H]
  const int32_t* token;  // [B][T]
  const int32_t* parent; // [T]
  const int32_t* paths;  // [NL][D+1]
  const int32_t* node_argmax;
  const float* node_lse;
  const float* node_entropy;
  const uint8_t* child_keep;  // typical keep flags from the verification merge, or null (computed here)
  const int32_t* bonus_src;   // [B][T] the token the bonus takes at the last kept node (node_argmax, or a draw)
  int32_t *accept_len, *acc_tokens, *acc_nodes, *bonus;
  uint8_t* ws;
};

template <typename TT>
__global__ void __launch_bounds__(256) accept_kernel(AcceptArgs a) {
  __shared__ unsigned char keep[MEDUSA_MAX_NODES];
  __shared__ int best_len[256], best_node[256], best_leaf[256];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* tok = a.token + (size_t)b * a.T;
  pdl_trigger();
  pdl_wait();

  if (!a.typical) {
    for (int c = 1 + threadIdx.x; c < a.T; c += blockDim.x)
      keep[c] = tok[c] == a.node_argmax[(size_t)b * a.T + a.parent[c]];
  } else if (a.child_keep) {
    for (int c = 1 + threadIdx.x; c < a.T; c += blockDim.x) keep[c] = a.child_keep[(size_t)b * a.T + c];
  } else {
    const TT* O = reinterpret_cast<const TT*>(a.attn_out);
    const TT* LM = reinterpret_cast<const TT*>(a.lm_head);
    for (int c = 1 + warp; c < a.T; c += blockDim.x / 32) {
      const int p = a.parent[c];
      const int t = tok[c];
      const bool t_ok = t >= 0 && t < a.V;
      float s = 0.f;
      if (t_ok)
        for (int j = lane; j < a.H; j += 32)
          s = fmaf(to_f32(LM[(size_t)t * a.H + j]), to_f32(O[((size_t)b * a.T + p) * a.H + j]), s);
      s = warp_sum(s);
      if (lane == 0) {
        if (!t_ok) set_error(a.ws, MEDUSA_ERR_DEVICE);
        const size_t pi = (size_t)b * a.T + p;
        const float logp = s * a.inv_temp - a.node_lse[pi];
        const float logthr = fminf(a.log_eps, a.log_delta - a.node_entropy[pi]);
        keep[c] = t_ok && (logp > logthr);
      }
    }
  }
  __syncthreads();

  // per leaf: the kept prefix of its path (rows of shallow leaves end in -1);
  // the longest wins, ties to the smaller last kept node, which in this node
  // order is the lower node at the first divergence; then the lower leaf
  int bl = -1, bnode = INT_MAX, bleaf = INT_MAX;
  for (int leaf = threadIdx.x; leaf < a.NL; leaf += blockDim.x) {
    const int32_t* path = a.paths + (size_t)leaf * (a.D + 1);
    int n = 0;
    while (n < a.D && path[n + 1] >= 0 && keep[path[n + 1]]) ++n;
    const int node = path[n];
    if (n > bl || (n == bl && node < bnode)) {  // leaves visited in increasing order
      bl = n;
      bnode = node;
      bleaf = leaf;
    }
  }
  best_len[threadIdx.x] = bl;
  best_node[threadIdx.x] = bnode;
  best_leaf[threadIdx.x] = bleaf;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      const int ol = best_len[threadIdx.x + s], on = best_node[threadIdx.x + s], of = best_leaf[threadIdx.x + s];
      const int ml = best_len[threadIdx.x], mn = best_node[threadIdx.x], mf = best_leaf[threadIdx.x];
      if (ol > ml || (ol == ml && (on < mn || (on == mn && of < mf)))) {
        best_len[threadIdx.x] = ol;
        best_node[threadIdx.x] = on;
        best_leaf[threadIdx.x] = of;
      }
    }
    __syncthreads();
  }
  const int n = best_len[0], leaf = best_leaf[0];
  const int32_t* path = a.paths + (size_t)leaf * (a.D + 1);
  for (int d = threadIdx.x; d <= a.D; d += blockDim.x) {
    a.acc_nodes[(size_t)b * (a.D + 1) + d] = d <= n ? path[d] : -1;
    if (d < a.D) a.acc_tokens[(size_t)b * a.D + d] = d < n ? tok[path[d + 1]] : -1;
  }
  if (threadIdx.x == 0) {
    a.accept_len[b] = n;
    a.bonus[b] = a.bonus_src[(size_t)b * a.T + path[n]];
  }
}

int launch_accept(const Plan& p, const void* attn_out, const void* lm_head, const medusa_tree_t& t,
                  const int32_t* node_argmax, const float* node_lse, const float* node_entropy, int32_t* accept_len,
                  int32_t* acc_tokens, int32_t* acc_nodes, int32_t* bonus, uint8_t* ws, cudaStream_t st) {
  AcceptArgs a;
  a.B = p.B;
  a.T = p.T;
  a.D = p.D;
  a.NL = p.NL;
  a.V = p.V;
  a.H = p.H;
  a.typical = p.typical ? 1 : 0;
  a.inv_temp = p.typical ? 1.f / p.temperature : 1.f;
  a.log_eps = logf(p.eps);
  a.log_delta = p.delta > 0.f ? logf(p.delta) : -INFINITY;
  a.attn_out = attn_out;
  a.lm_head = lm_head;
  a.token = t.token;
  a.parent = t.parent;
  a.paths = t.paths;
  a.node_argmax = node_argmax;
  a.node_lse = node_lse;
  a.node_entropy = node_entropy;
  a.child_keep = p.typical && (p.bf16 || p.sharded) ? ws + p.off_keep : nullptr;
  a.bonus_src = p.sample_bonus ? reinterpret_cast<const int32_t*>(ws + p.off_draw) : node_argmax;
  a.accept_len = accept_len;
  a.acc_tokens = acc_tokens;
  a.acc_nodes = acc_nodes;
  a.bonus = bonus;
  a.ws = ws;
  if (p.bf16) return (int)launch_k(accept_kernel<__nv_bfloat16>, dim3(p.B), dim3(256), 0, st, true, a);
  return (int)launch_k(accept_kernel<float>, dim3(p.B), dim3(256), 0, st, true, a);
}

// bf16: tensor-core projection; fp32 (no TF32 anywhere): the CUDA-core stream kernel
int launch_verify(const Plan& p, const void* attn_out, const void* lm_head, const int32_t* token, int32_t* node_argmax,
                  float* node_maxlogit, float* node_lse, float* node_entropy, uint8_t* ws, cudaStream_t st) {
  if (p.bf16)
    return launch_verify_tc(p, attn_out, lm_head, token, node_argmax, node_maxlogit, node_lse, node_entropy, ws, st);
  return launch_verify_rows(p, attn_out, lm_head, node_argmax, node_maxlogit, node_lse, node_entropy, ws, st);
}

int launch_verify_accept(const Plan& p, const void* attn_out, const void* lm_head, const medusa_tree_t& t,
                         int32_t* node_argmax, float* node_maxlogit, float* node_lse, float* node_entropy,
                         int32_t* accept_len, int32_t* acc_tokens, int32_t* acc_nodes, int32_t* bonus, uint8_t* ws,
                         cudaStream_t st) {
  int e = launch_verify(p, attn_out, lm_head, t.token, node_argmax, node_maxlogit, node_lse, node_entropy, ws, st);
  if (e) return e;
  return launch_accept(p, attn_out, lm_head, t, node_argmax, node_lse, node_entropy, accept_len, acc_tokens,
                       acc_nodes, bonus, ws, st);
}

}  // namespace medusa
