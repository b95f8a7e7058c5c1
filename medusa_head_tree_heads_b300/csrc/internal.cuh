// Internal declarations shared by the translation units of libmedusa.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/medusa.h"

namespace medusa {

constexpr int kThreads = 256;   // threads per CTA of the streaming kernels
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPieces = 4;   // segments one streaming CTA may touch
constexpr int kMaxStreamCtas = 1024;  // cap of the persistent streaming grids (workspace sizing)
constexpr int kHeadsTcMaxCtas = 160;  // cap of the tensor-core heads grids (one CTA per SM)
constexpr int kHeadsTcMaxBatch = 32;  // largest batch of the tensor-core heads (projection N = 2B <= 64)

// ---------------------------------------------------------------- workspace --
// [0, 256): int32 error word at 0, tickets from word 8 on.
enum Ticket { TICKET_FC = 8, TICKET_PROJ = 9, TICKET_VERIFY = 10,
              TICKET_PROJ_DONE = 11,    // medusa_step: projection CTAs finished this step
              TICKET_ATTN_DONE = 12 };  // overlap schedule: tree attention CTAs finished this step

// The candidate tree as tables, filled on the host for the Cartesian tree of
// the per-depth list sizes or for a caller's explicit tree.  Nodes are in
// (depth, parent, rank) order with node 0 the root, so a node's children are
// consecutive.  Kernels take them in their grid-constant parameters.
struct TreeDims {
  int T, n_leaves, W, D;
  int16_t parent[MEDUSA_MAX_NODES];       // -1 for the root
  uint8_t depth[MEDUSA_MAX_NODES];
  uint8_t rank[MEDUSA_MAX_NODES];         // rank in the head list of the node's depth (root 0)
  int16_t first_child[MEDUSA_MAX_NODES];  // first child (children are consecutive), -1 for a leaf
  uint8_t n_child[MEDUSA_MAX_NODES];
  int16_t leaf[MEDUSA_MAX_NODES];         // leaf ids, increasing
};

struct Plan {
  // sizes
  int B, H, V, K, D, kmax, T, NL, W, Hq, Hkv, G, Dh, L, Lc;
  int Vs, v0;  // vocabulary rows this call holds (W2 per head, lm_head) and the id of its first row
  bool bf16, typical, sample;
  bool sample_bonus;  // typical acceptance whose bonus is a draw (MEDUSA_ACCEPT_TYPICAL_SAMPLE)
  float temperature, eps, delta;
  uint32_t seed[2];
  int step;
  TreeDims tree;
  int topk_n[MEDUSA_MAX_HEADS];  // entries kept per head
  // streaming partitions
  int sm_count;
  int heads_ctas;  // grid cap of the tensor-core heads kernels
  int schedule;    // medusa_schedule_t as given
  bool overlap;    // medusa_step only: tree attention beside the head projection
  bool late_tree;  // medusa_step only: candidate merge + tree beside the verification projection
  bool sharded;    // the config names a vocabulary shard (vocab_rows > 0)
  int fc_nc, fc_ctiles, pj_nc, pj_ctiles, vf_nc, vf_ctiles;  // columns per CTA, column tiles
  // workspace offsets (bytes)
  size_t off_z, off_cand_val, off_cand_idx, off_cand_seg, off_vf_part, off_vf_idx, off_vtc_part, off_attn_part;
  size_t off_zs, off_ht_slot, off_ht_tickets;  // tensor-core heads: z pairs, cut-tile partials, tickets
  size_t off_keep;  // [B][T] uint8 typical-acceptance keep flags written by the verification merge
  size_t off_draw_part, off_draw;  // typical with a sampled bonus: per-tile draws [n_vt][B*T] float2, draws [B*T]
  size_t total;
};

int make_plan(const medusa_config_t* cfg, Plan* p);  // medusa_status_t
void finish_plan(Plan* p);                            // launch shapes for the current device
// the two launches of the heads stage (shape-dependent kernel choice)
int launch_head_layer(const Plan& p, const void* h, const void* W1, const void* b1, uint8_t* ws, cudaStream_t st);
int launch_head_proj(const Plan& p, const void* W2, int32_t* topk_idx, float* topk_val, uint8_t* ws,
                     cudaStream_t st);
size_t verify_tc_part_bytes(int V, int N);
size_t heads_tc_zs_bytes(int K, int B, int H);
size_t heads_tc_slot_bytes(int B);
bool heads_tc_supported(const Plan& p);  // from make_plan's fields alone
int launch_fc_tc(const Plan& p, const void* h, const void* W1, const void* b1, uint8_t* ws, cudaStream_t st);
int launch_proj_tc_only(const Plan& p, const void* W2, uint8_t* ws, cudaStream_t st, int* ctas, int* upc, int* ups);
int launch_proj_tc(const Plan& p, const void* W2, int32_t* topk_idx, float* topk_val, uint8_t* ws, cudaStream_t st);
size_t attn_part_bytes(int B, int T, int G, int Hkv, int L, int Dh);
void attn_split_shape(int B, int T, int G, int Hkv, int L, int* NS, int* chunk_blks);
// the verification's two launches: the projection (partials per vocabulary
// tile) and the merge of the partials (node results, typical keep flags; or,
// for a vocabulary shard, the merged state per node into shard_out)
enum VerifyPart { VERIFY_BOTH = 0, VERIFY_GEMM = 1, VERIFY_MERGE = 2, VERIFY_SHARD = 3 };
int launch_verify_tc(const Plan& p, const void* attn_out, const void* lm_head, const int32_t* token, int32_t* node_argmax,
                     float* node_maxlogit, float* node_lse, float* node_entropy, uint8_t* ws, cudaStream_t st,
                     VerifyPart part = VERIFY_BOTH, float4* shard_out = nullptr);
int launch_merge_tree(const Plan& p, int32_t* topk_idx, float* topk_val, const int32_t* root,
                      const medusa_tree_t& t, uint8_t* ws, int nctas, int rpc, int S, bool count_wait,
                      cudaStream_t st);

// fp32 (or bf16 beyond the tensor-core kernels) verification on the CUDA
// cores; with soft_out the merged state per node goes there instead of the
// node results (a vocabulary shard)
int launch_verify_rows(const Plan& p, const void* attn_out, const void* lm_head, int32_t* node_argmax,
                       float* node_maxlogit, float* node_lse, float* node_entropy, uint8_t* ws, cudaStream_t st,
                       float4* soft_out = nullptr);

// Exchange record of one vocabulary shard (medusa_shard_partial writes it,
// medusa_shard_finish reads n of them back to back); offsets in bytes, every
// section 16-byte aligned:
//   0         int32 header {vocab_begin, vocab_rows, B*T, kmax}
//   off_val   float [B][K][kmax]  the shard's per-head top-k values (-inf pad)
//   off_idx   int32 [B][K][kmax]  their global token ids (-1 pad)
//   off_node  float4 [B*T]        per node: max score, sum e, sum e*t (typical),
//                                 argmax id bits (see shard_node_states)
//   off_cdot  float [B*T][kmax]   typical only: lm_head[idx] . o_node for the
//                                 shard's candidates of the node's child depth
struct ShardRecord {
  size_t off_val, off_idx, off_node, off_cdot, bytes;
};
ShardRecord shard_record_layout(const Plan& p);

// launchers (enqueue only; return cudaError_t as int)
int launch_heads(const Plan& p, const void* h, const void* W1, const void* b1, const void* W2, int32_t* topk_idx,
                 float* topk_val, uint8_t* ws, cudaStream_t st);
// head projection on the CUDA cores (streaming row kernel); with ctas / rpc
// the per-CTA top-k candidates stay in the workspace for the caller's merge
int launch_proj_topk(const Plan& p, const void* W2, int32_t* topk_idx, float* topk_val, uint8_t* ws,
                     cudaStream_t st, int* ctas = nullptr, int* rpc = nullptr);
int launch_tree_build(const Plan& p, const int32_t* topk_idx, const int32_t* root, const medusa_tree_t& t,
                      cudaStream_t st);
int attn_tc_splits(int B, int T, int G, int Hkv, int L);
bool attn_tc_supported(const Plan& p);
long long attn_tc_unsplit_ctas(const Plan& p);  // CTAs of the tensor-core attention without key splits
int heads_tc_proj_grid(const Plan& p);          // CTAs of the tensor-core head projection
int launch_tree_attn_tc(const Plan& p, const void* q, const void* kt, const void* vt, const void* kc, const void* vc,
                        const int32_t* lens, void* out, uint8_t* ws, cudaStream_t st);
int launch_tree_attn_mma(const Plan& p, const void* q, const void* kt, const void* vt, const void* kc, const void* vc,
                         const int32_t* lens, void* out, uint8_t* ws, cudaStream_t st);
int launch_tree_attn(const Plan& p, const void* q, const void* kt, const void* vt, const void* kc, const void* vc,
                     const int32_t* lens, void* out, uint8_t* ws, cudaStream_t st);
int launch_kv_commit(const Plan& p, const int32_t* acc_nodes, const int32_t* accept_len, const void* kt,
                     const void* vt, void* kc, void* vc, int32_t* lens, uint8_t* ws, cudaStream_t st);
int launch_next_inputs(const Plan& p, const void* attn_out, const int32_t* acc_nodes, const int32_t* accept_len,
                       const int32_t* bonus, void* h_next, int32_t* root_next, uint8_t* ws, cudaStream_t st);
int launch_verify_accept(const Plan& p, const void* attn_out, const void* lm_head, const medusa_tree_t& t,
                         int32_t* node_argmax, float* node_maxlogit, float* node_lse, float* node_entropy,
                         int32_t* accept_len, int32_t* acc_tokens, int32_t* acc_nodes, int32_t* bonus, uint8_t* ws,
                         cudaStream_t st);

// ------------------------------------------------------------ device helpers --
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// streaming 16-byte load that bypasses L1 (weights are read exactly once)
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Programmatic dependent launch.  Every kernel of the step calls pdl_trigger()
// on entry, so the next kernel in the stream may be scheduled onto SMs this
// one frees (its prologue overlaps this kernel's tail), and pdl_wait() before
// touching anything an earlier kernel of the stream writes or reads: that wait
// returns once the preceding grid has completed and its memory is visible.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// first error wins
__device__ __forceinline__ void set_error(uint8_t* ws, int code) {
  atomicCAS(reinterpret_cast<int*>(ws), 0, code);
}

// Bounded wait for a count that CTAs of an already running earlier grid raise
// (each after a fence over its outputs): one thread polls with acquire loads;
// past `budget_ns` it records MEDUSA_ERR_TIMEOUT and gives up.  The caller
// makes the rest of its CTA wait on that thread (a barrier).
__device__ __forceinline__ void wait_count(const int* count, int target, uint64_t budget_ns, uint8_t* ws) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
    if (v >= target) return;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > budget_ns) {
      set_error(ws, MEDUSA_ERR_TIMEOUT);
      return;
    }
  }
}

// Makes the data an acquire (wait_count) has seen visible to the reads of the
// async proxy (TMA loads) that follow in this thread.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// float -> int with the same order (negative floats have their magnitude bits flipped)
__device__ __forceinline__ int order_key(float x) {
  const int b = __float_as_int(x);
  return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float order_key_inv(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

// cache rows of sequence b: its own length when a per-sequence array is
// given (a value outside [0, Lc] is a device error and is clamped), else L
__device__ __forceinline__ int seq_len(const int32_t* lens, int b, int L, int Lc, uint8_t* ws) {
  if (!lens) return L;
  const int l = lens[b];
  if (l < 0 || l > Lc) {
    set_error(ws, MEDUSA_ERR_DEVICE);
    return l < 0 ? 0 : Lc;
  }
  return l;
}

// (value desc, index asc) order used by every top-k / argmax
__device__ __forceinline__ bool better(float v, int i, float w, int j) { return v > w || (v == w && i < j); }

}  // namespace medusa
