// medusa_heads_topk_noalloc: the heads + per-head top-k stage for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they run the heads: a serving loop whose allocator is frozen
// after warm-up, code running under a memory budget that forbids new
// allocations, or a host runtime that owns no CUDA allocator at all.  They can
// still pass their inputs and outputs, but not a workspace.  This entry point
// therefore keeps the stage's scratch -- the fp32 head activations z and the
// per-CTA top-k candidates -- in one fixed array compiled into the library.
//
// Limits and sharing:
//   * the array holds kNoAllocScratchBytes (16 MiB) on every GPU that loads
//     the library, until the process exits.  The heads stage gets its own
//     compact layout inside it (error word and tickets, then z, the top-k
//     candidates and, for the tensor-core heads, the z pairs, cut-tile
//     partials and their tickets): nothing of the later stages is counted.
//     A config whose heads scratch is larger is rejected with
//     MEDUSA_ERR_UNSUPPORTED before any launch;
//   * every call on a device uses the same array and leaves its contents
//     behind, and the layout moves with the config, so stale data of an
//     earlier call (another config, or a kernel that gave up on a bounded
//     wait) can sit anywhere.  Each call therefore clears everything that
//     must start at zero before its kernels run: the error word and the
//     streaming tickets, and both ticket arrays of the tensor-core heads;
//   * calls whose work overlaps on the GPU (other streams, other host
//     threads) race on the array: serialise them;
//   * device-side error codes land in the array's error word, which this
//     entry point does not report.
// The array's device address is looked up once per device with
// cudaGetSymbolAddress, on the first call made with that device current;
// make that first call before any stream capture.
#include <mutex>

#include "internal.cuh"

namespace medusa {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
constexpr int kHeadsTickets = 2 * kHeadsTcMaxCtas;  // the layer's and the projection's boundary tickets
static void* g_scratch_addr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of the scratch array for the current device (set-up on first use).
static int scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MEDUSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MEDUSA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
  return MEDUSA_OK;
}

static bool al16(const void* x) { return x && ((uintptr_t)x & 15u) == 0; }
static size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Offsets of the heads stage alone, packed from byte 256 on (the first 256
// bytes hold the error word and the tickets); returns the end.  The kernels
// read every offset from the plan, so a plan laid out here runs unchanged.
static size_t heads_only_layout(Plan* p) {
  size_t o = 256;
  const bool tc = heads_tc_supported(*p);
  p->off_z = o;
  if (!tc) o = up256(o + (size_t)p->B * p->K * p->H * sizeof(float));  // fp32 z of the streaming layer
  const size_t n_cand = (size_t)kMaxStreamCtas * kMaxPieces * p->B * p->kmax;
  p->off_cand_val = o;
  o = up256(o + n_cand * sizeof(float));
  p->off_cand_idx = o;
  o = up256(o + n_cand * sizeof(int));
  p->off_cand_seg = o;
  o = up256(o + (size_t)kMaxStreamCtas * kMaxPieces * sizeof(int));
  p->off_zs = p->off_ht_slot = p->off_ht_tickets = o;
  if (tc) {
    p->off_zs = o;
    o = up256(o + heads_tc_zs_bytes(p->K, p->B, p->H));
    p->off_ht_slot = o;
    o = up256(o + heads_tc_slot_bytes(p->B));
    p->off_ht_tickets = o;
    o = up256(o + kHeadsTickets * sizeof(int));
  }
  p->total = o;
  return o;
}

}  // namespace medusa

using namespace medusa;

extern "C" int medusa_heads_topk_noalloc(const medusa_config_t* cfg, const void* h, const void* W1, const void* b1,
                                         const void* W2, int32_t* topk_idx, float* topk_val, void* stream) {
  Plan p;
  int s = make_plan(cfg, &p);
  if (s != MEDUSA_OK) return s;
  if (!al16(h) || !al16(W1) || !al16(b1) || !al16(W2) || !topk_idx || !topk_val || p.sharded)
    return MEDUSA_ERR_INVALID_ARG;
  const bool tc = heads_tc_supported(p);
  if (heads_only_layout(&p) > kNoAllocScratchBytes) return MEDUSA_ERR_UNSUPPORTED;
  uint8_t* ws = nullptr;
  if ((s = scratch_for_current_device(&ws)) != MEDUSA_OK) return s;
  finish_plan(&p);
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return MEDUSA_ERR_CUDA;  // error word + tickets
  if (tc && cudaMemsetAsync(ws + p.off_ht_tickets, 0, kHeadsTickets * sizeof(int), st) != cudaSuccess)
    return MEDUSA_ERR_CUDA;
  int e = launch_head_layer(p, h, W1, b1, ws, st);
  if (e) return MEDUSA_ERR_CUDA;
  e = launch_head_proj(p, W2, topk_idx, topk_val, ws, st);
  return e ? MEDUSA_ERR_CUDA : MEDUSA_OK;
}
