/*
 * medusa.h -- C ABI of libmedusa.so: one Medusa speculative decode step on a
 * B300 (sm_103a).
 *
 * The step (sources: "Medusa Heads", ultralytics glossary, sections "Come le
 * teste prevedono i token successivi" and "Attenzione sull'albero e
 * accettazione"; "Tetes de decodage Medusa", aiunderstanding.org, section
 * "Plongee profonde"; arXiv 2401.10774, abstract):
 *   1. K Medusa heads read the final hidden state h:
 *        z_k = h + SiLU(W1_k h + b1_k),  logits_k = W2_k z_k
 *      and each keeps its top-k tokens                    -> medusa_heads_topk
 *   2. the per-depth top-k lists are combined by Cartesian product into a
 *      prefix-sharing candidate tree whose attention mask lets a node see
 *      only its ancestors (and itself)                    -> medusa_tree_build
 *   3. all tree nodes attend, in one pass, to the KV cache and to their
 *      ancestors                                           -> medusa_tree_attn
 *   4. the base lm_head scores every node; the longest branch the base model
 *      agrees with is kept (greedy: candidate == top choice; typical: the
 *      candidate's probability exceeds an entropy-tied threshold)
 *                                                          -> medusa_verify_accept
 *   medusa_step runs 1-4 in order on one stream.
 *
 * Conventions
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller allocates and owns all memory (inputs, outputs, the tree arrays
 *     and the workspace).  The library allocates nothing per call.
 *   - All tensors are dense row-major in the layouts given below; the
 *     floating-point tensors use the config's dtype (fp32 or bf16) unless a
 *     type is named; pointers to bf16/fp32 tensors must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  A non-zero return means nothing was enqueued (host
 *     validation failed) or a launch failed.  Faults detected on the device
 *     (an index out of range, a bounded wait that ran out) set an error word
 *     in the workspace, read with medusa_get_device_error.
 *   - The workspace (medusa_workspace_bytes) must be zero-filled once after
 *     allocation; every call leaves it ready for the next one.  Calls that
 *     share a workspace must not overlap on the GPU.
 *
 * Symbols: B batch, H hidden, V vocab, K heads, D tree depth, k_d top-k at
 * depth d, T = 1 + sum_d prod_{j<=d} k_j tree nodes (root included),
 * NL = prod_d k_d leaves, W = ceil(T/32) mask words per node, L kv_len,
 * Lc kv_capacity, Hq/Hkv query/kv heads, Dh head dim (Hq*Dh == H).
 */
#ifndef MEDUSA_H
#define MEDUSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MEDUSA_MAX_DEPTH 8   /* D <= 8 */
#define MEDUSA_MAX_HEADS 8   /* K <= 8 */
#define MEDUSA_MAX_TOPK 16   /* k_d <= 16 */
#define MEDUSA_MAX_NODES 512 /* T <= 512 */

typedef enum {
  MEDUSA_OK = 0,
  MEDUSA_ERR_INVALID_ARG = -1, /* null/misaligned pointer, inconsistent sizes */
  MEDUSA_ERR_UNSUPPORTED = -2, /* sizes outside the limits above */
  MEDUSA_ERR_CUDA = -3,        /* a CUDA launch or runtime call failed */
  MEDUSA_ERR_TIMEOUT = -4,     /* device: a bounded wait ran out */
  MEDUSA_ERR_DEVICE = -5       /* device: an index check failed */
} medusa_status_t;

typedef enum { MEDUSA_F32 = 0, MEDUSA_BF16 = 1 } medusa_dtype_t;
/* GREEDY: keep a candidate equal to its parent's top choice.  TYPICAL: keep a
 * candidate whose probability clears an entropy-tied threshold.  SAMPLE: each
 * node's choice is a draw from its distribution at the temperature (Gumbel-max
 * with counter-based noise, see medusa_verify_accept); a candidate equal to
 * its parent's draw is kept, so the accepted tokens follow the base model's
 * sampling distribution (bf16 only).  This is rejection sampling against the
 * base model over the tree's fixed candidates ("Tetes de decodage Medusa":
 * exact rejection sampling keeps the base model's distribution): trying the
 * children in rank order, each accepted with its probability renormalised
 * over the tokens not yet rejected, and drawing the bonus from the rest, emits
 * the same distribution; one draw per node decides all of it at once.
 * TYPICAL_SAMPLE: typical acceptance whose bonus token is that draw at the
 * last kept node instead of the top choice (bf16 only; not with vocabulary
 * shards). */
typedef enum {
  MEDUSA_ACCEPT_GREEDY = 0,
  MEDUSA_ACCEPT_TYPICAL = 1,
  MEDUSA_ACCEPT_SAMPLE = 2,
  MEDUSA_ACCEPT_TYPICAL_SAMPLE = 3
} medusa_accept_t;
/* Launch order of medusa_step (the results are the same bits either way).
 * SERIAL: heads, candidate tree, tree attention, verification, acceptance.
 * OVERLAP: the tree attention runs beside the head projection, on the SMs the
 * projection's grid leaves free (the attention reads no head output); bf16,
 * head dim 128 and B <= 32 only, else MEDUSA_ERR_UNSUPPORTED.  AUTO takes
 * OVERLAP wherever it is supported (measured as fast or faster at every
 * supported shape tried, e.g. the 7B-shaped step 293 us against 301 us),
 * else SERIAL.  With the tensor-core heads (bf16,
 * B <= 32) both orders issue the verification projection before the
 * candidate merge and tree, which then run beside it.  Any other value is
 * MEDUSA_ERR_INVALID_ARG (every call validates the config). */
typedef enum { MEDUSA_SCHEDULE_AUTO = 0, MEDUSA_SCHEDULE_SERIAL = 1, MEDUSA_SCHEDULE_OVERLAP = 2 } medusa_schedule_t;

/* Sizes and options of one step (host memory, read during the call only). */
typedef struct {
  int32_t batch;                   /* B >= 1 */
  int32_t hidden;                  /* H, a multiple of 64 */
  int32_t vocab;                   /* V >= 2 */
  int32_t n_heads;                 /* K, depth <= K <= 8 */
  int32_t depth;                   /* D, 0 <= D <= 8 */
  int32_t topk[MEDUSA_MAX_DEPTH];  /* k_1..k_D, 1 <= k_d <= 16, k_d <= V */
  int32_t n_q_heads;               /* Hq */
  int32_t n_kv_heads;              /* Hkv, Hq % Hkv == 0 */
  int32_t head_dim;                /* Dh in {64, 128}; Hq*Dh == H */
  int32_t kv_len;                  /* L >= 0 valid cache rows per sequence */
  int32_t kv_capacity;             /* Lc >= L: cache rows allocated per sequence */
  int32_t dtype;                   /* medusa_dtype_t of weights/activations */
  int32_t accept_mode;             /* medusa_accept_t */
  float temperature;               /* typical, sample: softmax temperature (> 0) */
  float eps;                       /* typical: threshold cap */
  float delta;                     /* typical: threshold scale, thr = min(eps, delta*exp(-H)) */
  /* Optional explicit candidate tree ("Medusa Heads", "Attenzione sull'albero
   * e accettazione" speaks of the tree built from the heads' candidates; a
   * sparse subset of the Cartesian product is the same structure with fewer
   * branches).  0 = the Cartesian tree of topk[].  Otherwise tree_nodes = T
   * nodes in strictly increasing (depth, parent, rank) order, node 0 the root:
   * tree_parent[i] < i (-1 for node 0), node depth = parent depth + 1 <= depth,
   * tree_rank[i] < topk[depth - 1] (0 for the root).  Host arrays, read during
   * the call only; anything else is MEDUSA_ERR_INVALID_ARG (T > 512:
   * MEDUSA_ERR_UNSUPPORTED). */
  int32_t tree_nodes;
  const int32_t* tree_parent;
  const int32_t* tree_rank;
  /* SAMPLE, TYPICAL_SAMPLE: the noise of vocabulary row v at node n = b*T + i is drawn
   * from Philox4x32-10 with key (sample_seed[0], sample_seed[1]) and counter
   * (v, n / 4, sample_step, 0), word n % 4; a new step needs a new
   * sample_step (or seed). */
  uint32_t sample_seed[2];
  int32_t sample_step;
  int32_t schedule; /* medusa_schedule_t, read by medusa_step and medusa_step_launches */
  /* Vocabulary shard (medusa_shard_partial only; see there): this call's W2
   * holds rows [vocab_begin, vocab_begin + vocab_rows) of every head, as
   * [K][vocab_rows][H], and its lm_head the same rows, as [vocab_rows][H];
   * token ids stay global (0 .. vocab - 1).  vocab_rows = 0: the whole
   * vocabulary, which every other entry point requires (else
   * MEDUSA_ERR_INVALID_ARG).  Needs max_d k_d <= vocab_rows. */
  int32_t vocab_begin;
  int32_t vocab_rows;
} medusa_config_t;

/* Candidate tree, device arrays allocated by the caller (sizes from
 * medusa_tree_size).  Nodes are numbered breadth first: node 0 is the root;
 * depth-d nodes follow depth-(d-1) nodes, ordered by parent then by rank in
 * the head-d list.  Leaves are the nodes without children, in increasing
 * order; a leaf shallower than the tree depth ends its path row with -1. */
typedef struct {
  int32_t* token;   /* [B][T] candidate token; token[b][0] = root_token[b] */
  int32_t* parent;  /* [T] parent node, -1 for the root */
  int32_t* depth;   /* [T] */
  int32_t* rank;    /* [T] rank of the node's token in its head's list (root 0) */
  uint32_t* mask;   /* [T][W] bit j of word j/32 set iff node j is node i or an ancestor */
  int32_t* paths;   /* [NL][D+1] node ids from the root to each leaf, then -1 */
  int32_t* pos;     /* [T] position id kv_len + depth */
} medusa_tree_t;

/* All tensors of one fused step (device pointers). */
typedef struct {
  /* inputs */
  const void* h;           /* [B][H] final hidden state */
  const void* W1;          /* [K][H][H] head layer weight (out, in) */
  const void* b1;          /* [K][H] head layer bias */
  const void* W2;          /* [K][V][H] head vocabulary projection */
  const void* lm_head;     /* [V][H] base model output layer */
  const int32_t* root_token; /* [B] base model's token for the next position */
  const void* q;           /* [B][T][Hq][Dh] tree queries */
  const void* k_tree;      /* [B][T][Hkv][Dh] tree keys */
  const void* v_tree;      /* [B][T][Hkv][Dh] tree values */
  const void* k_cache;     /* [B][Lc][Hkv][Dh] cache keys (rows < L are read) */
  const void* v_cache;     /* [B][Lc][Hkv][Dh] cache values */
  /* outputs */
  int32_t* topk_idx;       /* [B][K][kmax] see medusa_heads_topk */
  float* topk_val;         /* [B][K][kmax] */
  medusa_tree_t tree;      /* see medusa_tree_build */
  void* attn_out;          /* [B][T][H] see medusa_tree_attn */
  int32_t* node_argmax;    /* [B][T] see medusa_verify_accept */
  float* node_maxlogit;    /* [B][T] */
  float* node_lse;         /* [B][T] typical only (may be NULL for greedy) */
  float* node_entropy;     /* [B][T] typical only (may be NULL for greedy) */
  int32_t* accept_len;     /* [B] */
  int32_t* acc_tokens;     /* [B][D] */
  int32_t* acc_nodes;      /* [B][D+1] */
  int32_t* bonus;          /* [B] */
  /* optional: per-sequence cache lengths (device [B], each in [0, kv_capacity];
   * the config's kv_len still sizes the key splits).  NULL: kv_len for all.
   * Cache rows past a sequence's length must hold finite values (e.g. zeros
   * from allocation): their keys are masked and their values weighted 0. */
  const int32_t* kv_lens;
} medusa_step_io_t;

/* Bytes of device workspace the calls below need for this config (0 on an
 * invalid config).  Host-only. */
size_t medusa_workspace_bytes(const medusa_config_t* cfg);

/* Tree sizes for this config: T nodes, NL leaves, W mask words per node.
 * Host-only; any output pointer may be NULL.  Returns a medusa_status_t. */
int medusa_tree_size(const medusa_config_t* cfg, int32_t* n_nodes, int32_t* n_leaves, int32_t* mask_words);

/* Heads and per-head top-k ("Medusa Heads", "Come le teste prevedono i token
 * successivi": each head is a residual SiLU feed-forward layer followed by a
 * vocabulary projection; "Attenzione sull'albero e accettazione": the best
 * tokens of each head form the tree).
 *   z_k = h + SiLU(W1_k h + b1_k) (fp32, in the workspace), logits_k = W2_k z_k.
 *   topk_idx[b][k][r], topk_val[b][k][r]: rank r of head k, descending logit,
 *   ties to the lower token id; kmax = max_d k_d; head k (0-based) keeps
 *   k_{k+1} entries when k < D, else 1; unused entries are -1 / -inf.
 * h [B][H], W1 [K][H][H], b1 [K][H], W2 [K][V][H].
 * Kernels: bf16 batches of at most 32 sequences run both head matrices on the
 * tensor cores (z kept as a bf16 hi/lo pair, about 16 significant bits);
 * larger bf16 batches and every fp32 config stream the weights through the
 * CUDA cores (fp32 z and accumulation).  The results agree within the
 * stated tolerances either way; only the speed differs (the CUDA-core path
 * runs at 2B multiply-adds per weight element and falls below the memory
 * bound as B grows). */
int medusa_heads_topk(const medusa_config_t* cfg, const void* h, const void* W1, const void* b1,
                      const void* W2, int32_t* topk_idx, float* topk_val, void* workspace, void* stream);

/* Cartesian candidate tree ("Attenzione sull'albero e accettazione": the
 * product of the heads' lists, shared prefixes, ancestor-only mask).  Writes
 * every array of *tree (the struct itself is host memory).  token[b][i] =
 * topk_idx[b][depth_i - 1][rank_i]. */
int medusa_tree_build(const medusa_config_t* cfg, const int32_t* topk_idx, const int32_t* root_token,
                      const medusa_tree_t* tree, void* stream);

/* medusa_heads_topk without a caller workspace, for callers that cannot
 * allocate device memory (a frozen allocator in a serving loop, a memory
 * budget that forbids new allocations, a host runtime with no CUDA
 * allocator).  It has no counterpart in the method's description: it exists
 * only for this calling constraint.  Same inputs, outputs and results as
 * medusa_heads_topk; the scratch lives in a fixed 16 MiB device array inside
 * the library (held on every GPU that loads it until exit), so a config that
 * needs more returns MEDUSA_ERR_UNSUPPORTED.  All calls on a device share that
 * array -- calls that overlap on the GPU race, so serialise them.  The first
 * call on a device looks up the array's address (make it before any stream
 * capture).  Device-side error codes are not reported by this variant. */
int medusa_heads_topk_noalloc(const medusa_config_t* cfg, const void* h, const void* W1, const void* b1,
                              const void* W2, int32_t* topk_idx, float* topk_val, void* stream);

/* Tree attention in one pass ("Attenzione sull'albero e accettazione"; "Plongee
 * profonde"): for each b, q head h (kv head h / (Hq/Hkv)) and node i,
 *   o = sum_j softmax_j(q.k_j / sqrt(Dh)) v_j
 * over the L cache rows and the tree nodes j with mask[i] bit j.
 * attn_out [B][T][H] holds o of q head h at columns h*Dh .. h*Dh+Dh-1, in the
 * config's dtype.  The ancestor-or-self relation (mask[i]) comes from the
 * config's tree (the tree built by medusa_tree_build for this config has the
 * same mask); the tree's device arrays are not read, tree->mask is only
 * checked to be present. */
int medusa_tree_attn(const medusa_config_t* cfg, const void* q, const void* k_tree, const void* v_tree,
                     const void* k_cache, const void* v_cache, const medusa_tree_t* tree, void* attn_out,
                     void* workspace, void* stream);

/* Verification and acceptance ("Attenzione sull'albero e accettazione").
 * Scores s_i = lm_head . attn_out[b][i] (fp32 accumulation) for every node:
 *   node_argmax (ties to the lower id), node_maxlogit; typical mode also
 *   node_lse = log sum_v exp(s_v / temperature) and node_entropy = -sum p ln p
 *   of p = softmax(s / temperature).  Sample mode: node_argmax = the argmax of
 *   s_v / temperature + g_v (a draw from softmax(s / temperature)), with
 *   Gumbel noise g_v = -ln(-ln u), u = (top 24 bits of the Philox word + 0.5)
 *   / 2^24, and node_maxlogit = that maximum.
 * Acceptance: an edge parent->c is kept when (greedy, sample) token_c ==
 * node_argmax[parent], or (typical) p_parent(token_c) > min(eps, delta *
 * exp(-entropy_parent)).  The longest chain of kept edges from the root wins
 * (ties: lowest node id at the first divergence).  accept_len[b] = its
 * length n; acc_tokens[b][0..n) its tokens; acc_nodes[b][0..n] its nodes
 * (root first); bonus[b] = node_argmax at its last node; unused entries -1.
 * Reads tree->token, tree->parent, tree->paths. */
int medusa_verify_accept(const medusa_config_t* cfg, const void* attn_out, const void* lm_head,
                         const medusa_tree_t* tree, int32_t* node_argmax, float* node_maxlogit, float* node_lse,
                         float* node_entropy, int32_t* accept_len, int32_t* acc_tokens, int32_t* acc_nodes,
                         int32_t* bonus, void* workspace, void* stream);

/* medusa_tree_attn with a per-sequence cache length kv_lens[b] (device [B],
 * each in [0, kv_capacity]; see medusa_step_io_t.kv_lens).  A length outside
 * that range sets MEDUSA_ERR_DEVICE and is clamped. */
int medusa_tree_attn_lens(const medusa_config_t* cfg, const void* q, const void* k_tree, const void* v_tree,
                          const void* k_cache, const void* v_cache, const int32_t* kv_lens,
                          const medusa_tree_t* tree, void* attn_out, void* workspace, void* stream);

/* KV commit: the accepted branch ("Attenzione sull'albero e accettazione": the
 * kept branch is appended and feeds the next round) moves into the cache.  For
 * each sequence b with n = accept_len[b]: the key and value rows of nodes
 * acc_nodes[b][0..n] (root first) are copied from k_tree / v_tree to cache rows
 * kv_lens[b] .. kv_lens[b] + n, then kv_lens[b] += n + 1 (device array, in and
 * out).  A node id outside the tree, n outside [0, depth] or a cache without
 * room sets MEDUSA_ERR_DEVICE and leaves that sequence unchanged.  The pages
 * give no such call; it is the step after acceptance. */
int medusa_kv_commit(const medusa_config_t* cfg, const int32_t* acc_nodes, const int32_t* accept_len,
                     const void* k_tree, const void* v_tree, void* k_cache, void* v_cache, int32_t* kv_lens,
                     void* workspace, void* stream);

/* Next-round inputs: h_next[b] ([B][H], config dtype) = attn_out[b][node] for the
 * last accepted node node = acc_nodes[b][accept_len[b]] (the tree output the
 * base lm_head read), root_next[b] = bonus[b].  Bad indices set
 * MEDUSA_ERR_DEVICE.  The pages give no such call; it is the step after. */
int medusa_next_inputs(const medusa_config_t* cfg, const void* attn_out, const int32_t* acc_nodes,
                       const int32_t* accept_len, const int32_t* bonus, void* h_next, int32_t* root_next,
                       void* workspace, void* stream);

/* The whole step: heads_topk, tree_build, tree_attn, verify_accept on
 * `stream`, in the order cfg->schedule picks (MEDUSA_SCHEDULE_OVERLAP issues
 * the tree attention right after the head projection, which it runs beside).
 * io is host memory holding device pointers.  Everything the step reads may be
 * written by earlier work in the stream, and everything it writes may be read
 * by later work: kernels of the step start early only beside other kernels of
 * the same step, and the first one waits for all earlier work.  With fp32
 * storage the tree attention and the verification run on a second stream of
 * the calling host thread (created on the first such call on each device
 * that is not inside a graph capture; until then, or if that fails, the step
 * runs in `stream` alone), forked from `stream` by an
 * event and joined back before the acceptance, so the ordering above holds
 * unchanged; inside a graph capture of `stream` this gives two branches. */
int medusa_step(const medusa_config_t* cfg, const medusa_step_io_t* io, void* workspace, void* stream);

/* medusa_step with timing: the same launches, plus an external event record
 * (cudaEventRecordExternal, so it also times correctly inside a captured CUDA
 * graph) of events[2k] just before and events[2k+1] just after stage k
 * (events: host array of n_events >= 2 * MEDUSA_STEP_KERNELS cudaEvent_t
 * created by the caller).  Stages, each one or two kernel launches: 0 head
 * layer, 1 head projection (at batch <= 32 with bf16 the tensor-core kernel
 * alone; otherwise with its top-k candidate merge), 2 tree build (at batch
 * <= 32 with bf16 fused with the top-k candidate merge), 3 tree attention
 * (+ split combine), 4 verification projection (+ partial merge),
 * 5 acceptance.  Under MEDUSA_SCHEDULE_OVERLAP stage 3 is issued before stage
 * 2 (the results are the same; its stage times may include overlap with the
 * projection).  With fp32 the profiled step does not fork (stages in order,
 * in `stream`; the top-k merge and the tree build are then two launches, one
 * in medusa_step), and its results equal medusa_step's bit for bit. */
#define MEDUSA_STEP_KERNELS 6
int medusa_step_profiled(const medusa_config_t* cfg, const medusa_step_io_t* io, void* workspace, void* stream,
                         void* const* events, int32_t n_events);

/* Number of kernel launches one medusa_step makes for this config on the
 * current device (the kernels chosen depend on the shape and the SM count);
 * negative medusa_status_t on an invalid config.  Host-only. */
int medusa_step_launches(const medusa_config_t* cfg);

/* Vocabulary-sharded step over several GPUs (one process per GPU; arXiv
 * 2401.10774, abstract: the step is memory-bound, so at batch 1 only a split
 * of the weights lowers the bytes each GPU reads).  GPU s of G holds rows
 * [vocab_begin, vocab_begin + vocab_rows) of every head projection and of
 * lm_head (cfg->vocab_begin / cfg->vocab_rows; the shards tile 0 .. vocab-1
 * in rank order).  A step is:
 *   medusa_shard_partial   on every GPU, writes its record
 *   (the caller)           all-gathers the records into one device buffer,
 *                          rank order, records back to back
 *   medusa_shard_finish    on every GPU, the same results as medusa_step
 * The top-k lists over the whole vocabulary are the top-k of the union of
 * the shards' lists; a node's argmax, maximum, log-partition and entropy
 * combine exactly from per-shard states; a child's typical-acceptance score
 * comes from the shard holding its token's row.  Host-only; 0 when the config
 * names no shard (vocab_rows = 0) or is invalid. */
size_t medusa_shard_record_bytes(const medusa_config_t* cfg);

/* This GPU's part of the step: heads and per-head top-k over its rows,
 * the sequence-independent tree arrays (parent, depth, rank, pos, mask,
 * paths: written into io->tree), tree attention of every node (io->attn_out,
 * replicated on every GPU; io->kv_lens as in medusa_step) and the
 * verification over its rows.  record (device, medusa_shard_record_bytes,
 * 16-byte aligned): int32 header {vocab_begin, vocab_rows, B*T, kmax}, the
 * shard's top-k values and global ids [B][K][kmax], per node the state
 * (max score, sum e, sum e*t, argmax id bits) with t = (score - max) /
 * temperature (typical; e = exp t), and for typical acceptance the scores
 * lm_head[id] . o_node of the shard's candidates of each node's child depth
 * [B*T][kmax].  io->W2 is [K][vocab_rows][H], io->lm_head [vocab_rows][H]; the
 * other inputs as in medusa_step; io's top-k, node and acceptance outputs are
 * not written.  A config without a shard is MEDUSA_ERR_INVALID_ARG. */
int medusa_shard_partial(const medusa_config_t* cfg, const medusa_step_io_t* io, void* record, void* workspace,
                         void* stream);

/* The combination: records = n_shards records back to back (device).  Writes
 * io's top-k lists (global), the tree's tokens and arrays, node_argmax,
 * node_maxlogit, (typical) node_lse / node_entropy and the acceptance
 * outputs, identical on every GPU.  Records that do not tile the vocabulary
 * in order set MEDUSA_ERR_DEVICE in the workspace error word.  Reads no
 * weight. */
int medusa_shard_finish(const medusa_config_t* cfg, const medusa_step_io_t* io, const void* records,
                        int32_t n_shards, void* workspace, void* stream);

/* Checks, on the current device, the bounded-wait path every kernel of the
 * library uses: one CTA waits on an mbarrier that nothing completes; after
 * budget_us microseconds (1..1000000) the wait gives up, MEDUSA_ERR_TIMEOUT
 * is recorded in the workspace error word and the kernel returns, leaving the
 * context usable.  Read the result with medusa_get_device_error. */
int medusa_check_bounded_wait(void* workspace, int32_t budget_us, void* stream);

/* Copies the device error word of `workspace` to *code (host pointer; 0 = no
 * error, else a medusa_status_t) after synchronising `stream`, then clears it. */
int medusa_get_device_error(void* workspace, int32_t* code, void* stream);

/* Human-readable name of a status code (static string). */
const char* medusa_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MEDUSA_H */
