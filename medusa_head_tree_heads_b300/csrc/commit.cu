// The steps on either side of the hot path ("Medusa Heads", "Attenzione
// sull'albero e accettazione": the kept branch is appended to the output and
// feeds the heads for the next round).
//
//   kv commit    the accepted path (root included: node ids acc_nodes[b][0..n],
//                n = accept_len[b]) moves from the tree's keys / values into
//                the cache at rows kv_lens[b] .. kv_lens[b] + n, and
//                kv_lens[b] grows by n + 1
//   next inputs  the next step's hidden state is the attention output at the
//                last accepted node (the tree output the base model's lm_head
//                read), and its root token is this step's bonus token
//
// Pure data movement: one CTA per sequence, 16-byte copies.  Bad indices or a
// full cache set MEDUSA_ERR_DEVICE and leave that sequence untouched.  Both
// kernels run only after everything before them in the stream (no
// programmatic early start), and the next kernel starts only after they end.
#include "internal.cuh"

namespace medusa {

struct CommitArgs {
  int B, T, D, Lc;
  int row_vec;  // 16-byte vectors per key/value row (Hkv * Dh elements)
  const int32_t* acc_nodes;   // [B][D+1]
  const int32_t* accept_len;  // [B]
  const uint4* kt;            // [B][T][row]
  const uint4* vt;
  uint4* kc;                  // [B][Lc][row]
  uint4* vc;
  int32_t* lens;              // [B] in/out
  uint8_t* ws;
};

__global__ void __launch_bounds__(256) kv_commit_kernel(CommitArgs a) {
  __shared__ int s_ok, s_l0, s_n;
  __shared__ int s_node[MEDUSA_MAX_DEPTH + 1];
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    const int n = a.accept_len[b], l0 = a.lens[b];
    bool ok = n >= 0 && n <= a.D && l0 >= 0 && l0 + n + 1 <= a.Lc;
    for (int d = 0; ok && d <= n; ++d) {
      const int node = a.acc_nodes[(size_t)b * (a.D + 1) + d];
      ok = node >= 0 && node < a.T;
      s_node[d] = node;
    }
    if (!ok) set_error(a.ws, MEDUSA_ERR_DEVICE);
    s_ok = ok;
    s_l0 = l0;
    s_n = n;
  }
  __syncthreads();
  if (!s_ok) return;
  const int n = s_n, l0 = s_l0;
  const int total = (n + 1) * a.row_vec;
  for (int e = threadIdx.x; e < total; e += blockDim.x) {
    const int d = e / a.row_vec, x = e - d * a.row_vec;
    const size_t src = ((size_t)b * a.T + s_node[d]) * a.row_vec + x;
    const size_t dst = ((size_t)b * a.Lc + l0 + d) * a.row_vec + x;
    a.kc[dst] = a.kt[src];
    a.vc[dst] = a.vt[src];
  }
  __syncthreads();
  if (threadIdx.x == 0) a.lens[b] = l0 + n + 1;
}

struct NextArgs {
  int T, D;
  int row_vec;  // 16-byte vectors per hidden row (H elements)
  const uint4* attn_out;      // [B][T][row]
  const int32_t* acc_nodes;   // [B][D+1]
  const int32_t* accept_len;  // [B]
  const int32_t* bonus;       // [B]
  uint4* h_next;              // [B][row]
  int32_t* root_next;         // [B]
  uint8_t* ws;
};

__global__ void __launch_bounds__(256) next_inputs_kernel(NextArgs a) {
  const int b = blockIdx.x;
  const int n = a.accept_len[b];
  const int node = (n >= 0 && n <= a.D) ? a.acc_nodes[(size_t)b * (a.D + 1) + n] : -1;
  if (node < 0 || node >= a.T) {
    if (threadIdx.x == 0) set_error(a.ws, MEDUSA_ERR_DEVICE);
    return;
  }
  for (int x = threadIdx.x; x < a.row_vec; x += blockDim.x)
    a.h_next[(size_t)b * a.row_vec + x] = a.attn_out[((size_t)b * a.T + node) * a.row_vec + x];
  if (threadIdx.x == 0) a.root_next[b] = a.bonus[b];
}

int launch_kv_commit(const Plan& p, const int32_t* acc_nodes, const int32_t* accept_len, const void* kt,
                     const void* vt, void* kc, void* vc, int32_t* lens, uint8_t* ws, cudaStream_t st) {
  CommitArgs a;
  a.B = p.B;
  a.T = p.T;
  a.D = p.D;
  a.Lc = p.Lc;
  a.row_vec = p.Hkv * p.Dh * (p.bf16 ? 2 : 4) / 16;
  a.acc_nodes = acc_nodes;
  a.accept_len = accept_len;
  a.kt = reinterpret_cast<const uint4*>(kt);
  a.vt = reinterpret_cast<const uint4*>(vt);
  a.kc = reinterpret_cast<uint4*>(kc);
  a.vc = reinterpret_cast<uint4*>(vc);
  a.lens = lens;
  a.ws = ws;
  kv_commit_kernel<<<p.B, 256, 0, st>>>(a);
  return (int)cudaGetLastError();
}

int launch_next_inputs(const Plan& p, const void* attn_out, const int32_t* acc_nodes, const int32_t* accept_len,
                       const int32_t* bonus, void* h_next, int32_t* root_next, uint8_t* ws, cudaStream_t st) {
  NextArgs a;
  a.T = p.T;
  a.D = p.D;
  a.row_vec = p.H * (p.bf16 ? 2 : 4) / 16;
  a.attn_out = reinterpret_cast<const uint4*>(attn_out);
  a.acc_nodes = acc_nodes;
  a.accept_len = accept_len;
  a.bonus = bonus;
  a.h_next = reinterpret_cast<uint4*>(h_next);
  a.root_next = root_next;
  a.ws = ws;
  next_inputs_kernel<<<p.B, 256, 0, st>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace medusa
