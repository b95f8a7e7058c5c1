// Vocabulary-sharded step: each GPU holds rows [v0, v0 + Vs) of every head
// projection and of lm_head.  The step is memory-bound (arXiv 2401.10774,
// abstract), so at batch 1 the bytes a GPU reads fall with its share of the
// rows; what the rows give is small and combines exactly:
//   * a head's top-k over the whole vocabulary is the top-k of the union of
//     the shards' top-k lists (ids are global, so ties still go to the lower
//     id);
//   * a node's argmax, maximum, log-partition and entropy come from per-shard
//     states (max, argmax, sum e, sum e*t with t the score minus the max, over
//     the temperature): the larger maximum wins and the sums are brought to it
//     (the same join the verification uses between vocabulary tiles);
//   * typical acceptance scores a child token under its parent's
//     distribution: the shard that holds the token's lm_head row computes that
//     dot product for each of its own candidates, and the combination keeps
//     the one whose candidate made the global list.
// medusa_shard_partial writes one record per shard (layout: ShardRecord in
// internal.cuh), the caller all-gathers the records, medusa_shard_finish
// combines them into the global lists, the tree, the node results and the
// acceptance (the same answer on every GPU).
#include <limits.h>

#include "internal.cuh"

namespace medusa {

int launch_topk_merge(const Plan& p, int32_t* topk_idx, float* topk_val, uint8_t* ws, int ctas, int rpc, int S,
                      cudaStream_t st);
int launch_accept(const Plan& p, const void* attn_out, const void* lm_head, const medusa_tree_t& t,
                  const int32_t* node_argmax, const float* node_lse, const float* node_entropy, int32_t* accept_len,
                  int32_t* acc_tokens, int32_t* acc_nodes, int32_t* bonus, uint8_t* ws, cudaStream_t st);

static size_t up16(size_t x) { return (x + 15) / 16 * 16; }

ShardRecord shard_record_layout(const Plan& p) {
  ShardRecord r;
  const size_t nl = (size_t)p.B * p.K * p.kmax, nn = (size_t)p.B * p.T;
  r.off_val = 16;
  r.off_idx = up16(r.off_val + nl * sizeof(float));
  r.off_node = up16(r.off_idx + nl * sizeof(int32_t));
  r.off_cdot = up16(r.off_node + nn * sizeof(float4));
  r.bytes = up16(r.off_cdot + (p.typical ? nn * p.kmax * sizeof(float) : 0));
  return r;
}

// ------------------------------------------------------------ shard side --
// Header, and (typical) per node n of depth d < D and candidate j of this
// shard's list for head d: cdot[n][j] = lm_head[idx - v0] . o_n, one warp per
// (node, candidate).
struct ShardTailArgs {
  int B, T, H, K, kmax, D, v0, Vs;
  int topk_n[MEDUSA_MAX_HEADS];
  TreeDims td;
  const void* attn_out;  // [B][T][H]
  const void* lm_head;   // [Vs][H] (this shard's rows)
  uint8_t* rec;
  ShardRecord lay;
  int typical;
  uint8_t* ws;
};

template <typename TT>
__global__ void __launch_bounds__(256) shard_tail_kernel(const __grid_constant__ ShardTailArgs a) {
  pdl_trigger();
  pdl_wait();  // the lists and the attention output come from earlier kernels
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    int32_t* hd = reinterpret_cast<int32_t*>(a.rec);
    hd[0] = a.v0;
    hd[1] = a.Vs;
    hd[2] = a.B * a.T;
    hd[3] = a.kmax;
  }
  if (!a.typical) return;
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= (long long)a.B * a.T * a.kmax) return;
  const int j = (int)(w % a.kmax);
  const int n = (int)(w / a.kmax);  // b * T + i
  const int b = n / a.T, i = n - b * a.T;
  const int d = a.td.depth[i];
  float* cdot = reinterpret_cast<float*>(a.rec + a.lay.off_cdot);
  int kn = 0;
#pragma unroll
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k)
    if (k == d) kn = a.topk_n[k];
  const int32_t* idx = reinterpret_cast<const int32_t*>(a.rec + a.lay.off_idx);
  const int t = (d < a.D && j < kn) ? idx[((size_t)b * a.K + d) * a.kmax + j] : -1;
  const int r = t - a.v0;
  float s = 0.f;
  if (t >= 0 && r >= 0 && r < a.Vs) {
    const TT* lm = reinterpret_cast<const TT*>(a.lm_head) + (size_t)r * a.H;
    const TT* o = reinterpret_cast<const TT*>(a.attn_out) + (size_t)n * a.H;
    for (int x = lane; x < a.H; x += 32) s = fmaf(to_f32(lm[x]), to_f32(o[x]), s);
  }
  s = warp_sum(s);
  if (lane == 0) cdot[(size_t)n * a.kmax + j] = (t >= 0) ? s : 0.f;
}

// ---------------------------------------------------------- combination --
struct ShardFinishArgs {
  TreeDims td;
  int B, K, kmax, T, L, V, n_shards;
  int topk_n[MEDUSA_MAX_HEADS];
  int typical;
  float inv_temp, log_eps, log_delta;
  const uint8_t* recs;  // n_shards records of lay.bytes each
  ShardRecord lay;
  const int32_t* root;  // [B]
  medusa_tree_t t;
  int32_t* out_idx;  // [B][K][kmax]
  float* out_val;
  int32_t* node_argmax;
  float* node_maxlogit;
  float* node_lse;
  float* node_entropy;
  uint8_t* keep;  // [B][T] typical keep flags (read by the acceptance)
  uint8_t* ws;
};

struct SState {
  float m, z, s;
  int i;
};

// join of two node states; z == 0 is empty (the same join the verification
// applies between vocabulary tiles)
__device__ __forceinline__ SState sjoin(const SState& a, const SState& b, bool typical, float it) {
  if (a.z == 0.f) return b;
  if (b.z == 0.f) return a;
  SState r;
  const bool af = better(a.m, a.i, b.m, b.i);
  r.m = af ? a.m : b.m;
  r.i = af ? a.i : b.i;
  if (typical) {
    const float da = (a.m - r.m) * it, db = (b.m - r.m) * it;
    const float ea = expf(da), eb = expf(db);
    r.z = a.z * ea + b.z * eb;
    r.s = ea * (a.s + a.z * da) + eb * (b.s + b.z * db);
  } else {
    r.z = a.z + b.z;
    r.s = 0.f;
  }
  return r;
}

// One CTA per sequence.  Warp k merges head k's lists of every shard (each
// lane a best-first list of its candidates, then kn rounds of "the best list
// head wins"), keeping where each winner came from; then the tree, the node
// results and (typical) the children's keep flags.
template <int KM>
__global__ void __launch_bounds__(256) shard_finish_kernel(const __grid_constant__ ShardFinishArgs a) {
  __shared__ int s_idx[MEDUSA_MAX_HEADS][MEDUSA_MAX_TOPK];
  __shared__ int s_src[MEDUSA_MAX_HEADS][MEDUSA_MAX_TOPK];  // shard << 8 | rank in that shard's list
  __shared__ int16_t s_parent[MEDUSA_MAX_NODES];
  __shared__ uint8_t s_depth[MEDUSA_MAX_NODES], s_rank[MEDUSA_MAX_NODES];
  __shared__ float s_lse[MEDUSA_MAX_NODES], s_ent[MEDUSA_MAX_NODES];
  const TreeDims& td = a.td;
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = td.T, W = td.W;
  pdl_trigger();
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    s_parent[i] = td.parent[i];
    s_depth[i] = td.depth[i];
    s_rank[i] = td.rank[i];
  }
  pdl_wait();  // the records (and the previous readers of every output) are done
  if (b == 0 && threadIdx.x == 0) {  // the shards must tile the vocabulary in rank order
    long long next = 0;
    for (int s = 0; s < a.n_shards; ++s) {
      const int32_t* hd = reinterpret_cast<const int32_t*>(a.recs + (size_t)s * a.lay.bytes);
      if (hd[0] != next || hd[1] < 1 || hd[2] != a.B * a.T || hd[3] != a.kmax) set_error(a.ws, MEDUSA_ERR_DEVICE);
      next = (long long)hd[0] + hd[1];
    }
    if (next != a.V) set_error(a.ws, MEDUSA_ERR_DEVICE);
  }
  if (warp < a.K) {
    const int k = warp;
    int kn = 1;
#pragma unroll
    for (int x = 0; x < MEDUSA_MAX_HEADS; ++x)
      if (x == k) kn = a.topk_n[x];
    float lv[KM];
    int li[KM], ls[KM];
#pragma unroll
    for (int x = 0; x < KM; ++x) {
      lv[x] = -INFINITY;
      li[x] = INT_MAX;
      ls[x] = -1;
    }
    for (int c = lane; c < a.n_shards * kn; c += 32) {
      const int s = c / kn, j = c - s * kn;
      const uint8_t* rec = a.recs + (size_t)s * a.lay.bytes;
      const size_t o = ((size_t)b * a.K + k) * a.kmax + j;
      float v = reinterpret_cast<const float*>(rec + a.lay.off_val)[o];
      int id = reinterpret_cast<const int32_t*>(rec + a.lay.off_idx)[o];
      int src = (s << 8) | j;
      if (id < 0) continue;
#pragma unroll
      for (int x = 0; x < KM; ++x) {  // compare-and-swap insertion, best first
        const bool sw = better(v, id, lv[x], li[x]);
        const float ov = lv[x];
        const int oi = li[x], os = ls[x];
        lv[x] = sw ? v : ov;
        li[x] = sw ? id : oi;
        ls[x] = sw ? src : os;
        v = sw ? ov : v;
        id = sw ? oi : id;
        src = sw ? os : src;
      }
    }
    for (int rnk = 0; rnk < a.kmax; ++rnk) {
      float bv = lv[0];
      int bi = li[0], bs = ls[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        const int os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
          bs = os;
        }
      }
      if (bi != INT_MAX && lv[0] == bv && li[0] == bi) {  // ids are unique: one owner pops
#pragma unroll
        for (int x = 0; x < KM - 1; ++x) {
          lv[x] = lv[x + 1];
          li[x] = li[x + 1];
          ls[x] = ls[x + 1];
        }
        lv[KM - 1] = -INFINITY;
        li[KM - 1] = INT_MAX;
        ls[KM - 1] = -1;
      }
      if (lane == 0) {
        const bool live = rnk < kn && bi != INT_MAX;
        const size_t o = ((size_t)b * a.K + k) * a.kmax + rnk;
        a.out_idx[o] = live ? bi : -1;
        a.out_val[o] = live ? bv : -INFINITY;
        s_idx[k][rnk] = live ? bi : -1;
        s_src[k][rnk] = live ? bs : -1;
      }
    }
  }
  // node states of this sequence: every shard's, joined
  const bool typical = a.typical != 0;
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    const size_t n = (size_t)b * T + i;
    SState m;
    m.m = -INFINITY;
    m.z = 0.f;
    m.s = 0.f;
    m.i = INT_MAX;
    for (int s = 0; s < a.n_shards; ++s) {
      const float4 q = reinterpret_cast<const float4*>(a.recs + (size_t)s * a.lay.bytes + a.lay.off_node)[n];
      SState o;
      o.m = q.x;
      o.z = q.y;
      o.s = q.z;
      o.i = __float_as_int(q.w);
      m = sjoin(m, o, typical, a.inv_temp);
    }
    a.node_argmax[n] = m.i;
    a.node_maxlogit[n] = m.m;
    if (typical) {
      const float lz = logf(m.z);
      s_lse[i] = m.m * a.inv_temp + lz;
      s_ent[i] = lz - m.s / m.z;
      a.node_lse[n] = s_lse[i];
      a.node_entropy[n] = s_ent[i];
    }
  }
  __syncthreads();
  // the tree: tokens of this sequence; the first CTA writes the
  // sequence-independent arrays
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    const int d = s_depth[i];
    a.t.token[(size_t)b * T + i] = d == 0 ? a.root[b] : s_idx[d - 1][s_rank[i]];
    if (typical && d > 0) {  // the child's score under its parent, from the shard that holds the token's row
      const int src = s_src[d - 1][s_rank[i]], p = s_parent[i];
      bool keep = false;
      if (src >= 0) {
        const uint8_t* rec = a.recs + (size_t)(src >> 8) * a.lay.bytes;
        const float cd = reinterpret_cast<const float*>(rec + a.lay.off_cdot)[((size_t)b * T + p) * a.kmax + (src & 255)];
        keep = cd * a.inv_temp - s_lse[p] > fminf(a.log_eps, a.log_delta - s_ent[p]);
      }
      a.keep[(size_t)b * T + i] = keep;
    }
    if (b == 0) {
      a.t.depth[i] = d;
      a.t.parent[i] = s_parent[i];
      a.t.rank[i] = s_rank[i];
      a.t.pos[i] = a.L + d;
    }
  }
  if (b == 0) {
    for (int e = threadIdx.x; e < T * W; e += blockDim.x) {  // mask word w of node i
      const int i = e / W, w = e - i * W;
      uint32_t word = 0;
      for (int j = i; j >= 0; j = s_parent[j])
        if ((j >> 5) == w) word |= 1u << (j & 31);
      a.t.mask[e] = word;
    }
    for (int l = threadIdx.x; l < td.n_leaves; l += blockDim.x) {  // root-to-leaf path, then -1
      const int leaf = td.leaf[l], dl = s_depth[leaf];
      int32_t* row = a.t.paths + (size_t)l * (td.D + 1);
      for (int d = td.D; d > dl; --d) row[d] = -1;
      for (int d = dl, j = leaf; d >= 0; --d, j = s_parent[j]) row[d] = j;
    }
  }
}

}  // namespace medusa

using namespace medusa;

static bool al16(const void* x) { return x && ((uintptr_t)x & 15u) == 0; }
static int cstat(int e) { return e == 0 ? MEDUSA_OK : MEDUSA_ERR_CUDA; }

extern "C" {

size_t medusa_shard_record_bytes(const medusa_config_t* cfg) {
  Plan p;
  if (make_plan(cfg, &p) != MEDUSA_OK || !p.sharded) return 0;
  return shard_record_layout(p).bytes;
}

int medusa_shard_partial(const medusa_config_t* cfg, const medusa_step_io_t* io, void* record, void* workspace,
                         void* stream) {
  if (!io) return MEDUSA_ERR_INVALID_ARG;
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!p.sharded) return MEDUSA_ERR_INVALID_ARG;
  if (p.sample_bonus) return MEDUSA_ERR_UNSUPPORTED;  // the record carries no draws
  const medusa_tree_t& t = io->tree;
  if (!al16(io->h) || !al16(io->W1) || !al16(io->b1) || !al16(io->W2) || !al16(io->lm_head) || !al16(io->q) ||
      !al16(io->k_tree) || !al16(io->v_tree) || !al16(io->attn_out) || !al16(record) || !al16(workspace) ||
      !t.token || !t.parent || !t.depth || !t.rank || !t.mask || !t.paths || !t.pos)
    return MEDUSA_ERR_INVALID_ARG;
  if ((p.L > 0 || (io->kv_lens && p.Lc > 0)) && (!al16(io->k_cache) || !al16(io->v_cache)))
    return MEDUSA_ERR_INVALID_ARG;
  finish_plan(&p);
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  uint8_t* rec = (uint8_t*)record;
  const ShardRecord lay = shard_record_layout(p);
  int32_t* lidx = reinterpret_cast<int32_t*>(rec + lay.off_idx);
  float* lval = reinterpret_cast<float*>(rec + lay.off_val);
  // heads over this shard's rows: the merged per-head lists go to the record
  int e = launch_head_layer(p, io->h, io->W1, io->b1, ws, st);
  if (!e) e = launch_head_proj(p, io->W2, lidx, lval, ws, st);
  // the sequence-independent tree arrays (the attention of some shapes reads
  // the mask), then the attention over every node, then the verification over
  // this shard's rows, its per-node states into the record
  if (!e) e = launch_tree_build(p, nullptr, nullptr, t, st);
  if (!e) e = launch_tree_attn(p, io->q, io->k_tree, io->v_tree, io->k_cache, io->v_cache, io->kv_lens, io->attn_out,
                               ws, st);
  float4* node = reinterpret_cast<float4*>(rec + lay.off_node);
  if (!e) {
    if (p.bf16) {
      e = launch_verify_tc(p, io->attn_out, io->lm_head, nullptr, nullptr, nullptr, nullptr, nullptr, ws, st,
                           VERIFY_GEMM);
      if (!e)
        e = launch_verify_tc(p, io->attn_out, io->lm_head, nullptr, nullptr, nullptr, nullptr, nullptr, ws, st,
                             VERIFY_SHARD, node);
    } else {
      e = launch_verify_rows(p, io->attn_out, io->lm_head, nullptr, nullptr, nullptr, nullptr, ws, st, node);
    }
  }
  if (!e) {
    ShardTailArgs a;
    a.B = p.B;
    a.T = p.T;
    a.H = p.H;
    a.K = p.K;
    a.kmax = p.kmax;
    a.D = p.D;
    a.v0 = p.v0;
    a.Vs = p.Vs;
    for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.topk_n[k] = p.topk_n[k];
    a.td = p.tree;
    a.attn_out = io->attn_out;
    a.lm_head = io->lm_head;
    a.rec = rec;
    a.lay = lay;
    a.typical = p.typical ? 1 : 0;
    a.ws = ws;
    const long long warps = p.typical ? (long long)p.B * p.T * p.kmax : 1;
    const dim3 grid((unsigned)((warps + 7) / 8));
    e = p.bf16 ? (int)launch_k(shard_tail_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, true, a)
               : (int)launch_k(shard_tail_kernel<float>, grid, dim3(256), 0, st, true, a);
  }
  return cstat(e);
}

int medusa_shard_finish(const medusa_config_t* cfg, const medusa_step_io_t* io, const void* records,
                        int32_t n_shards, void* workspace, void* stream) {
  if (!io) return MEDUSA_ERR_INVALID_ARG;
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!p.sharded || n_shards < 1 || n_shards > 255) return MEDUSA_ERR_INVALID_ARG;
  if (p.sample_bonus) return MEDUSA_ERR_UNSUPPORTED;
  const medusa_tree_t& t = io->tree;
  if (!al16(records) || !al16(workspace) || !io->root_token || !io->topk_idx || !io->topk_val ||
      !io->node_argmax || !io->node_maxlogit || !io->accept_len || !io->acc_tokens || !io->acc_nodes || !io->bonus ||
      !t.token || !t.parent || !t.depth || !t.rank || !t.mask || !t.paths || !t.pos)
    return MEDUSA_ERR_INVALID_ARG;
  if (p.typical && (!io->node_lse || !io->node_entropy)) return MEDUSA_ERR_INVALID_ARG;
  finish_plan(&p);
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  ShardFinishArgs a;
  a.td = p.tree;
  a.B = p.B;
  a.K = p.K;
  a.kmax = p.kmax;
  a.T = p.T;
  a.L = p.L;
  a.V = p.V;
  a.n_shards = n_shards;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.topk_n[k] = p.topk_n[k];
  a.typical = p.typical ? 1 : 0;
  a.inv_temp = (p.typical || p.sample) ? 1.f / p.temperature : 1.f;
  a.log_eps = p.typical ? logf(p.eps) : 0.f;
  a.log_delta = p.typical && p.delta > 0.f ? logf(p.delta) : -INFINITY;
  a.recs = (const uint8_t*)records;
  a.lay = shard_record_layout(p);
  a.root = io->root_token;
  a.t = t;
  a.out_idx = io->topk_idx;
  a.out_val = io->topk_val;
  a.node_argmax = io->node_argmax;
  a.node_maxlogit = io->node_maxlogit;
  a.node_lse = io->node_lse;
  a.node_entropy = io->node_entropy;
  a.keep = ws + p.off_keep;
  a.ws = ws;
  int e;
  if (p.kmax <= 4) e = (int)launch_k(shard_finish_kernel<4>, dim3(p.B), dim3(256), 0, st, true, a);
  else if (p.kmax <= 8) e = (int)launch_k(shard_finish_kernel<8>, dim3(p.B), dim3(256), 0, st, true, a);
  else e = (int)launch_k(shard_finish_kernel<MEDUSA_MAX_TOPK>, dim3(p.B), dim3(256), 0, st, true, a);
  if (e) return cstat(e);
  return cstat(launch_accept(p, io->attn_out, nullptr, t, io->node_argmax, io->node_lse, io->node_entropy,
                             io->accept_len, io->acc_tokens, io->acc_nodes, io->bonus, ws, st));
}

}  // extern "C"
