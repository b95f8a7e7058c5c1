// C ABI of libmedusa.so: argument validation, workspace layout, launch plan
// and the entry points declared in include/medusa.h.
#include <stdio.h>
#include <string.h>

#include "internal.cuh"

namespace medusa {

int launch_fc(const Plan& p, const void* h, const void* W1, const void* b1, uint8_t* ws, cudaStream_t st);
int launch_bounded_wait_probe(uint8_t* ws, uint64_t budget_ns, cudaStream_t st);

// head layer / head projection: the tensor-core kernel for bf16 batches up to
// 32, else the general streaming kernel
int launch_head_layer(const Plan& p, const void* h, const void* W1, const void* b1, uint8_t* ws,
                             cudaStream_t st) {
  if (heads_tc_supported(p)) return launch_fc_tc(p, h, W1, b1, ws, st);
  return launch_fc(p, h, W1, b1, ws, st);
}
int launch_head_proj(const Plan& p, const void* W2, int32_t* topk_idx, float* topk_val, uint8_t* ws,
                     cudaStream_t st);

int launch_verify(const Plan& p, const void* attn_out, const void* lm_head, const int32_t* token, int32_t* node_argmax,
                  float* node_maxlogit, float* node_lse, float* node_entropy, uint8_t* ws, cudaStream_t st);
int launch_accept(const Plan& p, const void* attn_out, const void* lm_head, const medusa_tree_t& t,
                  const int32_t* node_argmax, const float* node_lse, const float* node_entropy, int32_t* accept_len,
                  int32_t* acc_tokens, int32_t* acc_nodes, int32_t* bonus, uint8_t* ws, cudaStream_t st);

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int pick_nc(int H, int C) {
  int nc = 8;
  while (nc > 1 && ((size_t)nc * H * sizeof(float) > 64 * 1024 || nc / 2 >= C)) nc /= 2;
  return nc;
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

int make_plan(const medusa_config_t* c, Plan* p) {
  if (!c || !p) return MEDUSA_ERR_INVALID_ARG;
  memset(p, 0, sizeof(*p));
  if (c->batch < 1 || c->hidden < 64 || c->vocab < 2 || c->n_heads < 1 || c->depth < 0) return MEDUSA_ERR_INVALID_ARG;
  if (c->n_q_heads < 1 || c->n_kv_heads < 1 || c->kv_len < 0 || c->kv_capacity < c->kv_len)
    return MEDUSA_ERR_INVALID_ARG;
  if (c->dtype != MEDUSA_F32 && c->dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  if (c->accept_mode != MEDUSA_ACCEPT_GREEDY && c->accept_mode != MEDUSA_ACCEPT_TYPICAL &&
      c->accept_mode != MEDUSA_ACCEPT_SAMPLE && c->accept_mode != MEDUSA_ACCEPT_TYPICAL_SAMPLE)
    return MEDUSA_ERR_INVALID_ARG;
  if (c->accept_mode == MEDUSA_ACCEPT_SAMPLE && !(c->temperature > 0.f)) return MEDUSA_ERR_INVALID_ARG;
  if ((c->accept_mode == MEDUSA_ACCEPT_SAMPLE || c->accept_mode == MEDUSA_ACCEPT_TYPICAL_SAMPLE) &&
      c->dtype != MEDUSA_BF16)
    return MEDUSA_ERR_UNSUPPORTED;
  if (c->schedule != MEDUSA_SCHEDULE_AUTO && c->schedule != MEDUSA_SCHEDULE_SERIAL &&
      c->schedule != MEDUSA_SCHEDULE_OVERLAP)
    return MEDUSA_ERR_INVALID_ARG;
  if (c->schedule == MEDUSA_SCHEDULE_OVERLAP &&
      (c->dtype != MEDUSA_BF16 || c->head_dim != 128 || c->batch > kHeadsTcMaxBatch))
    return MEDUSA_ERR_UNSUPPORTED;  // needs the tensor-core heads and attention kernels
  if (c->n_heads > MEDUSA_MAX_HEADS || c->depth > MEDUSA_MAX_DEPTH || c->depth > c->n_heads)
    return MEDUSA_ERR_UNSUPPORTED;
  if (c->hidden % 64 != 0) return MEDUSA_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return MEDUSA_ERR_UNSUPPORTED;
  if ((long long)c->n_q_heads * c->head_dim != c->hidden || c->n_q_heads % c->n_kv_heads != 0)
    return MEDUSA_ERR_INVALID_ARG;
  if ((long long)c->n_heads * c->vocab > (1LL << 30) || (long long)c->n_heads * c->hidden > (1LL << 30))
    return MEDUSA_ERR_UNSUPPORTED;
  if ((c->accept_mode == MEDUSA_ACCEPT_TYPICAL || c->accept_mode == MEDUSA_ACCEPT_TYPICAL_SAMPLE) &&
      !(c->temperature > 0.f && c->eps > 0.f && c->delta >= 0.f))
    return MEDUSA_ERR_INVALID_ARG;
  if (c->vocab_rows < 0 || c->vocab_begin < 0 || (c->vocab_rows == 0 && c->vocab_begin != 0) ||
      (long long)c->vocab_begin + c->vocab_rows > c->vocab)
    return MEDUSA_ERR_INVALID_ARG;
  p->B = c->batch;
  p->H = c->hidden;
  p->V = c->vocab;
  p->Vs = c->vocab_rows ? c->vocab_rows : c->vocab;
  p->v0 = c->vocab_begin;
  p->sharded = c->vocab_rows > 0;
  p->K = c->n_heads;
  p->D = c->depth;
  p->Hq = c->n_q_heads;
  p->Hkv = c->n_kv_heads;
  p->G = c->n_q_heads / c->n_kv_heads;
  p->Dh = c->head_dim;
  p->L = c->kv_len;
  p->Lc = c->kv_capacity;
  p->bf16 = c->dtype == MEDUSA_BF16;
  p->typical = c->accept_mode == MEDUSA_ACCEPT_TYPICAL || c->accept_mode == MEDUSA_ACCEPT_TYPICAL_SAMPLE;
  p->sample = c->accept_mode == MEDUSA_ACCEPT_SAMPLE;
  p->sample_bonus = c->accept_mode == MEDUSA_ACCEPT_TYPICAL_SAMPLE;
  p->seed[0] = c->sample_seed[0];
  p->seed[1] = c->sample_seed[1];
  p->step = c->sample_step;
  p->temperature = c->temperature;
  p->eps = c->eps;
  p->delta = c->delta;
  p->schedule = c->schedule;
  // tree tables: the Cartesian tree of topk[] or the caller's explicit tree
  TreeDims& td = p->tree;
  td.D = p->D;
  p->kmax = 1;
  for (int d = 1; d <= p->D; ++d) {
    const int k = c->topk[d - 1];
    if (k < 1 || k > MEDUSA_MAX_TOPK || k > p->Vs) return MEDUSA_ERR_UNSUPPORTED;
    if (k > p->kmax) p->kmax = k;
  }
  int T = 0;
  if (c->tree_nodes == 0) {
    td.parent[0] = -1;
    td.depth[0] = 0;
    td.rank[0] = 0;
    T = 1;
    int lv0 = 0, lv1 = 1;  // nodes of the previous level
    for (int d = 1; d <= p->D; ++d) {
      const int lv2 = T;
      for (int par = lv0; par < lv1; ++par)
        for (int r = 0; r < c->topk[d - 1]; ++r) {
          if (T >= MEDUSA_MAX_NODES) return MEDUSA_ERR_UNSUPPORTED;
          td.parent[T] = (int16_t)par;
          td.depth[T] = (uint8_t)d;
          td.rank[T] = (uint8_t)r;
          ++T;
        }
      lv0 = lv2;
      lv1 = T;
    }
  } else {
    T = c->tree_nodes;
    if (T < 1 || T > MEDUSA_MAX_NODES) return MEDUSA_ERR_UNSUPPORTED;
    if (!c->tree_parent || !c->tree_rank) return MEDUSA_ERR_INVALID_ARG;
    if (c->tree_parent[0] != -1 || c->tree_rank[0] != 0) return MEDUSA_ERR_INVALID_ARG;
    td.parent[0] = -1;
    td.depth[0] = 0;
    td.rank[0] = 0;
    for (int i = 1; i < T; ++i) {
      const int par = c->tree_parent[i], r = c->tree_rank[i];
      if (par < 0 || par >= i) return MEDUSA_ERR_INVALID_ARG;
      const int d = td.depth[par] + 1;
      if (d > p->D || r < 0 || r >= c->topk[d - 1]) return MEDUSA_ERR_INVALID_ARG;
      // strictly increasing (depth, parent, rank): breadth-first, no repeated child
      const int pd = td.depth[i - 1], pp = td.parent[i - 1], pr = td.rank[i - 1];
      if (!(d > pd || (d == pd && (par > pp || (par == pp && r > pr))))) return MEDUSA_ERR_INVALID_ARG;
      td.parent[i] = (int16_t)par;
      td.depth[i] = (uint8_t)d;
      td.rank[i] = (uint8_t)r;
    }
  }
  td.T = T;
  td.n_leaves = 0;
  for (int i = 0; i < T; ++i) {
    td.first_child[i] = -1;
    td.n_child[i] = 0;
  }
  for (int i = 1; i < T; ++i) {
    const int par = td.parent[i];
    if (td.first_child[par] < 0) td.first_child[par] = (int16_t)i;
    td.n_child[par] += 1;
  }
  for (int i = 0; i < T; ++i)
    if (td.n_child[i] == 0) td.leaf[td.n_leaves++] = (int16_t)i;
  td.W = (td.T + 31) / 32;
  p->T = td.T;
  p->NL = td.n_leaves;
  p->W = td.W;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) p->topk_n[k] = k < p->D ? c->topk[k] : 1;
  if ((long long)p->B * p->T > (1LL << 24)) return MEDUSA_ERR_UNSUPPORTED;

  // workspace (sized for the largest grids the launch plan can pick)
  size_t o = 256;  // error word + tickets
  p->off_z = o;
  o = align_up(o + (size_t)p->B * p->K * p->H * sizeof(float), 256);
  const size_t n_cand = (size_t)kMaxStreamCtas * kMaxPieces * p->B * p->kmax;
  p->off_cand_val = o;
  o = align_up(o + n_cand * sizeof(float), 256);
  p->off_cand_idx = o;
  o = align_up(o + n_cand * sizeof(int), 256);
  p->off_cand_seg = o;
  o = align_up(o + (size_t)kMaxStreamCtas * kMaxPieces * sizeof(int), 256);
  const size_t n_vf = (size_t)kMaxStreamCtas * p->B * p->T;
  p->off_vf_part = o;
  o = align_up(o + n_vf * 3 * sizeof(float), 256);
  p->off_vf_idx = o;
  o = align_up(o + n_vf * sizeof(int), 256);
  p->off_vtc_part = o;
  if (p->bf16) o = align_up(o + verify_tc_part_bytes(p->Vs, p->B * p->T), 256);
  p->off_attn_part = o;
  if (p->bf16) o = align_up(o + attn_part_bytes(p->B, p->T, p->G, p->Hkv, p->L, p->Dh), 256);
  p->off_zs = p->off_ht_slot = p->off_ht_tickets = o;
  if (p->bf16 && p->B <= kHeadsTcMaxBatch) {  // the tensor-core heads may run (decided per device)
    p->off_zs = o;
    o = align_up(o + heads_tc_zs_bytes(p->K, p->B, p->H), 256);
    p->off_ht_slot = o;
    o = align_up(o + heads_tc_slot_bytes(p->B), 256);
    p->off_ht_tickets = o;
    o = align_up(o + 2 * kHeadsTcMaxCtas * sizeof(int), 256);
  }
  p->off_keep = o;
  o = align_up(o + (size_t)p->B * p->T, 256);
  p->off_draw_part = p->off_draw = o;
  if (p->sample_bonus) {
    p->off_draw_part = o;
    o = align_up(o + verify_tc_part_bytes(p->Vs, p->B * p->T) / 2, 256);  // float2 per (vocab tile, node)
    p->off_draw = o;
    o = align_up(o + (size_t)p->B * p->T * sizeof(int32_t), 256);
  }
  p->total = o;
  return MEDUSA_OK;
}

// launch shapes need the device's SM count
void finish_plan(Plan* p) {
  p->sm_count = sm_count();
  // The tensor-core heads kernels stream their weights faster on ~5/6 of the
  // SMs than on all of them (7B: 240 vs 252 us for layer + projection; 13B:
  // 306 vs 315), and on the SMs left over the tree attention's first CTAs
  // start early and run their key blocks during the projection (7B step: 316
  // vs 324 us).
  p->heads_ctas = p->sm_count - p->sm_count / 6;
  if (p->heads_ctas < 1) p->heads_ctas = 1;
  p->overlap = false;
  p->fc_nc = pick_nc(p->H, p->B);
  p->fc_ctiles = (p->B + p->fc_nc - 1) / p->fc_nc;
  p->pj_nc = pick_nc(p->H, p->B);
  p->pj_ctiles = (p->B + p->pj_nc - 1) / p->pj_nc;
  p->vf_nc = pick_nc(p->H, p->B * p->T);
  p->vf_ctiles = (p->B * p->T + p->vf_nc - 1) / p->vf_nc;
}

int launch_head_proj(const Plan& p, const void* W2, int32_t* topk_idx, float* topk_val, uint8_t* ws,
                     cudaStream_t st) {
  if (heads_tc_supported(p)) return launch_proj_tc(p, W2, topk_idx, topk_val, ws, st);
  return launch_proj_topk(p, W2, topk_idx, topk_val, ws, st);
}

static bool aligned16(const void* x) { return x && ((uintptr_t)x & 15u) == 0; }

// medusa_step's schedule (after finish_plan).  AUTO takes the overlap order
// wherever it is supported and the projection's grid leaves SMs free.
// Measured with the current kernels (first replays, before the power cap
// lowers the clock): 7B 293 us per step in the overlap order against 301 us in
// the serial one; 13B 478 against 482; GQA-76 1788 against 1811; the
// large-vocabulary GQA 1930-2002 against 1960; 33B 4297-4415 against
// 4438-4492.  (An earlier build had the last two 1% and 0.4% slower in the
// overlap order, when AUTO estimated the attention's time beside the
// projection and kept the serial order for them.)
static bool pick_overlap(const Plan& p) {
  if (p.schedule == MEDUSA_SCHEDULE_SERIAL) return false;
  if (!heads_tc_supported(p) || !attn_tc_supported(p)) return false;
  if (p.schedule == MEDUSA_SCHEDULE_OVERLAP) return true;
  return p.sm_count - heads_tc_proj_grid(p) >= 8;
}

static int cuda_status(int e) { return e == 0 ? MEDUSA_OK : MEDUSA_ERR_CUDA; }

static int check_tree(const Plan& p, const medusa_tree_t* t) {
  if (!t || !t->token || !t->parent || !t->depth || !t->rank || !t->mask || !t->paths || !t->pos)
    return MEDUSA_ERR_INVALID_ARG;
  return MEDUSA_OK;
}

}  // namespace medusa

using namespace medusa;

extern "C" {

size_t medusa_workspace_bytes(const medusa_config_t* cfg) {
  Plan p;
  if (make_plan(cfg, &p) != MEDUSA_OK) return 0;
  return p.total;
}

int medusa_tree_size(const medusa_config_t* cfg, int32_t* n_nodes, int32_t* n_leaves, int32_t* mask_words) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (n_nodes) *n_nodes = p.T;
  if (n_leaves) *n_leaves = p.NL;
  if (mask_words) *mask_words = p.W;
  return MEDUSA_OK;
}

int medusa_heads_topk(const medusa_config_t* cfg, const void* h, const void* W1, const void* b1, const void* W2,
                      int32_t* topk_idx, float* topk_val, void* workspace, void* stream) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!aligned16(h) || !aligned16(W1) || !aligned16(b1) || !aligned16(W2) || !topk_idx || !topk_val ||
      !aligned16(workspace) || p.sharded)
    return MEDUSA_ERR_INVALID_ARG;
  finish_plan(&p);
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  int e = launch_head_layer(p, h, W1, b1, ws, st);
  if (e) return cuda_status(e);
  return cuda_status(launch_head_proj(p, W2, topk_idx, topk_val, ws, st));
}

int medusa_tree_build(const medusa_config_t* cfg, const int32_t* topk_idx, const int32_t* root_token,
                      const medusa_tree_t* tree, void* stream) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!topk_idx || !root_token) return MEDUSA_ERR_INVALID_ARG;
  if ((s = check_tree(p, tree)) != MEDUSA_OK) return s;
  return cuda_status(launch_tree_build(p, topk_idx, root_token, *tree, (cudaStream_t)stream));
}

int medusa_tree_attn(const medusa_config_t* cfg, const void* q, const void* k_tree, const void* v_tree,
                     const void* k_cache, const void* v_cache, const medusa_tree_t* tree, void* attn_out,
                     void* workspace, void* stream) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(attn_out) || !tree || !tree->mask ||
      !aligned16(workspace))
    return MEDUSA_ERR_INVALID_ARG;
  if (p.L > 0 && (!aligned16(k_cache) || !aligned16(v_cache))) return MEDUSA_ERR_INVALID_ARG;
  finish_plan(&p);
  return cuda_status(launch_tree_attn(p, q, k_tree, v_tree, k_cache, v_cache, nullptr, attn_out,
                                      (uint8_t*)workspace, (cudaStream_t)stream));
}

int medusa_tree_attn_lens(const medusa_config_t* cfg, const void* q, const void* k_tree, const void* v_tree,
                          const void* k_cache, const void* v_cache, const int32_t* kv_lens,
                          const medusa_tree_t* tree, void* attn_out, void* workspace, void* stream) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(attn_out) || !tree || !tree->mask ||
      !kv_lens || !aligned16(workspace))
    return MEDUSA_ERR_INVALID_ARG;
  if (p.Lc > 0 && (!aligned16(k_cache) || !aligned16(v_cache))) return MEDUSA_ERR_INVALID_ARG;
  finish_plan(&p);
  return cuda_status(launch_tree_attn(p, q, k_tree, v_tree, k_cache, v_cache, kv_lens, attn_out,
                                      (uint8_t*)workspace, (cudaStream_t)stream));
}

int medusa_kv_commit(const medusa_config_t* cfg, const int32_t* acc_nodes, const int32_t* accept_len,
                     const void* k_tree, const void* v_tree, void* k_cache, void* v_cache, int32_t* kv_lens,
                     void* workspace, void* stream) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!acc_nodes || !accept_len || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !kv_lens || !aligned16(workspace))
    return MEDUSA_ERR_INVALID_ARG;
  return cuda_status(launch_kv_commit(p, acc_nodes, accept_len, k_tree, v_tree, k_cache, v_cache, kv_lens,
                                      (uint8_t*)workspace, (cudaStream_t)stream));
}

int medusa_next_inputs(const medusa_config_t* cfg, const void* attn_out, const int32_t* acc_nodes,
                       const int32_t* accept_len, const int32_t* bonus, void* h_next, int32_t* root_next,
                       void* workspace, void* stream) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!aligned16(attn_out) || !acc_nodes || !accept_len || !bonus || !aligned16(h_next) || !root_next ||
      !aligned16(workspace))
    return MEDUSA_ERR_INVALID_ARG;
  return cuda_status(launch_next_inputs(p, attn_out, acc_nodes, accept_len, bonus, h_next, root_next,
                                        (uint8_t*)workspace, (cudaStream_t)stream));
}

int medusa_verify_accept(const medusa_config_t* cfg, const void* attn_out, const void* lm_head,
                         const medusa_tree_t* tree, int32_t* node_argmax, float* node_maxlogit, float* node_lse,
                         float* node_entropy, int32_t* accept_len, int32_t* acc_tokens, int32_t* acc_nodes,
                         int32_t* bonus, void* workspace, void* stream) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!aligned16(attn_out) || !aligned16(lm_head) || !node_argmax || !node_maxlogit || !accept_len ||
      !acc_tokens || !acc_nodes || !bonus || !aligned16(workspace) || p.sharded)
    return MEDUSA_ERR_INVALID_ARG;
  if (p.typical && (!node_lse || !node_entropy)) return MEDUSA_ERR_INVALID_ARG;
  if ((s = check_tree(p, tree)) != MEDUSA_OK) return s;
  finish_plan(&p);
  return cuda_status(launch_verify_accept(p, attn_out, lm_head, *tree, node_argmax, node_maxlogit, node_lse,
                                          node_entropy, accept_len, acc_tokens, acc_nodes, bonus,
                                          (uint8_t*)workspace, (cudaStream_t)stream));
}

}  // extern "C"

namespace medusa {

// Validates every argument of the step, then launches its kernels in order,
// recording events[2k] / events[2k+1] around kernel k when events != NULL.
// A second stream of the calling host thread on the current device, with two
// events, for the step's fork (created on first use; none if creation fails,
// and the step then runs in one stream).  Per thread, so two host threads
// never record into each other's fork.  Never created while `capturing` (a
// stream or event creation could invalidate the caller's graph capture): that
// call runs in one stream.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool failed = false;
  ~SideStream() {  // at thread exit (errors ignored: the runtime may already be unloading)
    if (join) cudaEventDestroy(join);
    if (fork) cudaEventDestroy(fork);
    if (s) cudaStreamDestroy(s);
  }
};
static SideStream* side_stream(bool capturing) {
  constexpr int kMaxDevices = 64;
  thread_local SideStream per_dev[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = per_dev[dev];
  if (ss.failed) return nullptr;
  if (!ss.s && capturing) return nullptr;
  if (!ss.s) {
    if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      ss.failed = true;
      return nullptr;
    }
  }
  return &ss;
}

static int run_step(const medusa_config_t* cfg, const medusa_step_io_t* io, void* workspace, void* stream,
                    void* const* events, int n_events) {
  if (!io) return MEDUSA_ERR_INVALID_ARG;
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!aligned16(io->h) || !aligned16(io->W1) || !aligned16(io->b1) || !aligned16(io->W2) ||
      !aligned16(io->lm_head) || !io->root_token || !aligned16(io->q) || !aligned16(io->k_tree) ||
      !aligned16(io->v_tree) || !io->topk_idx || !io->topk_val || !aligned16(io->attn_out) || !io->node_argmax ||
      !io->node_maxlogit || !io->accept_len || !io->acc_tokens || !io->acc_nodes || !io->bonus ||
      !aligned16(workspace) || p.sharded)
    return MEDUSA_ERR_INVALID_ARG;
  if ((p.L > 0 || (io->kv_lens && p.Lc > 0)) && (!aligned16(io->k_cache) || !aligned16(io->v_cache)))
    return MEDUSA_ERR_INVALID_ARG;
  if (p.typical && (!io->node_lse || !io->node_entropy)) return MEDUSA_ERR_INVALID_ARG;
  if ((s = check_tree(p, &io->tree)) != MEDUSA_OK) return s;
  if (events && n_events < 2 * MEDUSA_STEP_KERNELS) return MEDUSA_ERR_INVALID_ARG;
  finish_plan(&p);
  p.overlap = pick_overlap(p);
  p.late_tree = heads_tc_supported(p);
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  int e = 0;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (events && cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MEDUSA_ERR_CUDA;
  auto rec = [&](int i) {  // inside a capture only external records keep their timestamps
    if (!events || e != 0) return;
    e = cap == cudaStreamCaptureStatusActive
            ? (int)cudaEventRecordWithFlags((cudaEvent_t)events[i], st, cudaEventRecordExternal)
            : (int)cudaEventRecord((cudaEvent_t)events[i], st);
  };
#define MEDUSA_STAGE(k, call) \
  rec(2 * (k));               \
  if (e == 0) e = (call);     \
  rec(2 * (k) + 1);           \
  if (e) return cuda_status(e);
#define MEDUSA_ATTN_STAGE                                                                                    \
  MEDUSA_STAGE(3, launch_tree_attn(p, io->q, io->k_tree, io->v_tree, io->k_cache, io->v_cache, io->kv_lens, \
                                   io->attn_out, ws, st))
  // CUDA-core path without stage events: the tree attention (its ancestor
  // masks built from the plan's parent table, not from the tree outputs) and
  // the verification (the rows kernel's needs no tokens) read none of the
  // heads' or the tree build's outputs, so they run on a second stream beside
  // the head layer, projection and tree build, and the acceptance waits for
  // both branches (inside a graph capture: two parallel branches)
  SideStream* side = nullptr;
  if (!events && !p.bf16 && !p.late_tree) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return MEDUSA_ERR_CUDA;
    side = side_stream(cs != cudaStreamCaptureStatusNone);
  }
  if (side) {
    e = (int)cudaEventRecord(side->fork, st);
    if (e) return cuda_status(e);
    int es = (int)cudaStreamWaitEvent(side->s, side->fork, 0);
    if (es == 0)
      es = launch_tree_attn(p, io->q, io->k_tree, io->v_tree, io->k_cache, io->v_cache, io->kv_lens, io->attn_out,
                            ws, side->s);
    if (es == 0)
      es = launch_verify(p, io->attn_out, io->lm_head, io->tree.token, io->node_argmax, io->node_maxlogit,
                         io->node_lse, io->node_entropy, ws, side->s);
    // the join is recorded and waited on even after a failed launch, so that
    // later work in `stream` never runs beside this step's second branch
    const int ej = (int)cudaEventRecord(side->join, side->s);
    // the heads branch: layer, projection, then one kernel for the top-k merge and the tree
    int ctas = 0, rpc = 0;
    e = launch_head_layer(p, io->h, io->W1, io->b1, ws, st);
    if (e == 0) e = launch_proj_topk(p, io->W2, io->topk_idx, io->topk_val, ws, st, &ctas, &rpc);
    if (e == 0)
      e = launch_merge_tree(p, io->topk_idx, io->topk_val, io->root_token, io->tree, ws, ctas, rpc, p.Vs, false, st);
    const int ew = ej == 0 ? (int)cudaStreamWaitEvent(st, side->join, 0) : ej;
    if (e == 0) e = es;
    if (e == 0) e = ew;
    if (e == 0)
      e = launch_accept(p, io->attn_out, io->lm_head, io->tree, io->node_argmax, io->node_lse, io->node_entropy,
                        io->accept_len, io->acc_tokens, io->acc_nodes, io->bonus, ws, st);
    return e ? cuda_status(e) : MEDUSA_OK;
  }
  MEDUSA_STAGE(0, launch_head_layer(p, io->h, io->W1, io->b1, ws, st))
  if (p.late_tree) {
    // Tensor-core heads: the projection, the tree attention and the
    // verification projection, none of which reads the candidate tree's
    // tokens, then the candidate merge + tree, which waits for the
    // projection's completion count and so runs beside the verification
    // projection, then the verification merge and the acceptance.
    int ctas = 0, upc = 0, ups = 0;
    MEDUSA_STAGE(1, launch_proj_tc_only(p, io->W2, ws, st, &ctas, &upc, &ups))
    MEDUSA_ATTN_STAGE
    MEDUSA_STAGE(4, launch_verify_tc(p, io->attn_out, io->lm_head, io->tree.token, io->node_argmax,
                                     io->node_maxlogit, io->node_lse, io->node_entropy, ws, st, VERIFY_GEMM))
    MEDUSA_STAGE(2, launch_merge_tree(p, io->topk_idx, io->topk_val, io->root_token, io->tree, ws, ctas, upc, ups,
                                      true, st))
    rec(10);
    if (e == 0)
      e = launch_verify_tc(p, io->attn_out, io->lm_head, io->tree.token, io->node_argmax, io->node_maxlogit,
                           io->node_lse, io->node_entropy, ws, st, VERIFY_MERGE);
    if (e == 0)
      e = launch_accept(p, io->attn_out, io->lm_head, io->tree, io->node_argmax, io->node_lse, io->node_entropy,
                        io->accept_len, io->acc_tokens, io->acc_nodes, io->bonus, ws, st);
    rec(11);
    if (e) return cuda_status(e);
    return MEDUSA_OK;
  }
  MEDUSA_STAGE(1, launch_head_proj(p, io->W2, io->topk_idx, io->topk_val, ws, st))
  MEDUSA_STAGE(2, launch_tree_build(p, io->topk_idx, io->root_token, io->tree, st))
  MEDUSA_ATTN_STAGE
  MEDUSA_STAGE(4, launch_verify(p, io->attn_out, io->lm_head, io->tree.token, io->node_argmax, io->node_maxlogit, io->node_lse,
                             io->node_entropy, ws, st))
  MEDUSA_STAGE(5, launch_accept(p, io->attn_out, io->lm_head, io->tree, io->node_argmax, io->node_lse,
                             io->node_entropy, io->accept_len, io->acc_tokens, io->acc_nodes, io->bonus, ws, st))
#undef MEDUSA_ATTN_STAGE
#undef MEDUSA_STAGE
  return MEDUSA_OK;
}

}  // namespace medusa

extern "C" {

int medusa_step(const medusa_config_t* cfg, const medusa_step_io_t* io, void* workspace, void* stream) {
  return run_step(cfg, io, workspace, stream, nullptr, 0);
}

int medusa_step_profiled(const medusa_config_t* cfg, const medusa_step_io_t* io, void* workspace, void* stream,
                         void* const* events, int32_t n_events) {
  if (!events) return MEDUSA_ERR_INVALID_ARG;
  return run_step(cfg, io, workspace, stream, events, n_events);
}

int medusa_check_bounded_wait(void* workspace, int32_t budget_us, void* stream) {
  if (!aligned16(workspace) || budget_us < 1 || budget_us > 1000000) return MEDUSA_ERR_INVALID_ARG;
  return cuda_status(launch_bounded_wait_probe((uint8_t*)workspace, (uint64_t)budget_us * 1000,
                                               (cudaStream_t)stream));
}

int medusa_step_launches(const medusa_config_t* cfg) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (p.sharded) return MEDUSA_ERR_INVALID_ARG;
  finish_plan(&p);
  p.overlap = pick_overlap(p);
  int n = 6;                                     // one launch per stage
  if (p.bf16 && !heads_tc_supported(p)) n += 1;  // separate top-k merge (else fused with the tree;
                                                 // fp32 forks, with the merge and the tree in one kernel)
  if (p.bf16) {
    int NS, cb;
    attn_split_shape(p.B, p.T, p.G, p.Hkv, p.L, &NS, &cb);
    if (attn_tc_supported(p)) NS = p.overlap ? 1 : attn_tc_splits(p.B, p.T, p.G, p.Hkv, p.L);
    if (NS > 1) n += 1;             // split-attention combine
    n += 1;                         // verification partial merge
  }
  return n;
}

int medusa_get_device_error(void* workspace, int32_t* code, void* stream) {
  if (!workspace || !code) return MEDUSA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MEDUSA_ERR_CUDA;
  *code = v;
  if (v != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), st) != cudaSuccess) return MEDUSA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MEDUSA_ERR_CUDA;
  }
  return MEDUSA_OK;
}

const char* medusa_status_string(int status) {
  switch (status) {
    case MEDUSA_OK: return "MEDUSA_OK";
    case MEDUSA_ERR_INVALID_ARG: return "MEDUSA_ERR_INVALID_ARG";
    case MEDUSA_ERR_UNSUPPORTED: return "MEDUSA_ERR_UNSUPPORTED";
    case MEDUSA_ERR_CUDA: return "MEDUSA_ERR_CUDA";
    case MEDUSA_ERR_TIMEOUT: return "MEDUSA_ERR_TIMEOUT";
    case MEDUSA_ERR_DEVICE: return "MEDUSA_ERR_DEVICE";
    default: return "MEDUSA_ERR_UNKNOWN";
  }
}

}  // extern "C"
