// libmoe: C ABI of the B300 MoE routing-and-expert step.
//
// This file is the only translation unit of the library: it includes every
// kernel, validates arguments on the host, and enqueues the launches.  The
// declarations and their contracts are in include/moe.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <string>

#include "../../include/moe.h"
#include "combine.cuh"
#include "common.cuh"
#include "dispatch.cuh"
#include "front.cuh"
#include "ffn.cuh"
#include "ffn_pair.cuh"
#include "ffn_fused.cuh"
#include "ffn_small.cuh"
#include "replica_copy.cuh"
#include "replicate.cuh"
#include "route.cuh"
#include "stats.cuh"

#define MOE_VERSION_STRING "moe-b300 0.1 (sm_103a)"

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

moe_status cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return MOE_OK;
  return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

moe_status cuda_at(const char* who, cudaError_t e, const char* where) {
  if (e == cudaSuccess) return MOE_OK;
  return fail(MOE_ERR_CUDA, "%s: %s: %s", who, where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool init = false;
  int num_sms = 0;
  bool ffn_attr[4] = {false, false, false, false};    // GeLU, SwiGLU, store, combine
  bool pair_attr[4] = {false, false, false, false};
  bool small_attr[4] = {false, false, false, false};
  int pair_clusters[4] = {0, 0, 0, 0};  // max co-resident CTA pairs per pair-kernel instance
  bool fused_attr[2] = {false, false};
  int fused_clusters[2] = {0, 0};    // max co-resident CTA pairs of the fused kernel (GeLU, SwiGLU)
  // The FFN's small-batch kernels run as a second chain on this stream, forked
  // from and joined back to the caller's stream (created once, kept for the
  // life of the process).
  cudaStream_t side = nullptr;
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
};

// Library options (moe_set_option).
// Process-wide and atomic: a call reads each option once when it is made.
std::atomic<int> g_opt_ffn_kernel{MOE_FFN_KERNEL_AUTO};
std::atomic<int> g_opt_ffn_selftest{0};  // one-shot: next GEMM1 withholds an accumulator signal
std::atomic<int> g_opt_ffn_small_sms{0};  // SM split of the FFN's small-batch path (0: none, -1: model)
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
std::mutex g_side_mu;  // one fork/join sequence at a time per process

moe_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device id %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e, "cudaDeviceGetAttribute");
    e = cudaStreamCreateWithFlags(&d.side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.fork_ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.join_ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_status(e, "device set-up (FFN side stream)");
    d.init = true;
  }
  *out = &d;
  return MOE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

moe_status get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return MOE_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return MOE_OK;
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// box of box_inner x box_outer, 128-byte swizzle (or none: rows of the box
// packed in shared memory), zero fill out of bounds.
moe_status encode_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                     uint32_t box_outer, bool swizzle = true) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MOE_OK;
}

// 3-D view of a weight matrix [rows][n] bf16 (n a multiple of 64) for the
// grouped kernels: dims (64, rows, n/64), strides (n*2, 128) bytes, box
// (64, 64, chunks), 128-byte swizzle.  One box brings `chunks` adjacent
// 64-column chunks of 64 rows, laid out in shared memory as `chunks` 2-D
// boxes of 64 x 64 one after another -- the layout the kernels' descriptors
// expect -- with one TMA request instead of `chunks`.
moe_status encode_w3d(CUtensorMap* m, const void* ptr, uint64_t n, uint64_t rows, uint32_t chunks) {
  cuuint64_t dims[3] = {64, rows, n / 64};
  cuuint64_t strides[2] = {n * 2, 128};
  cuuint32_t box[3] = {64, 64, chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
  return MOE_OK;
}

// Upper bound on the 256-row blocks of the fused FFN kernel: each unit (at
// most 2E of them) adds at most one partial block.
long long ffn_blocks_bound(long long A, int G) { return (A + 255) / 256 + (long long)G + 1; }

size_t ffn_inter_bytes(long long A, int F) {
  // bf16 intermediate [A, F], 1024-byte aligned
  return (((size_t)A * (size_t)F * 2 + 1023) / 1024) * 1024;
}

// G: group count of the call (2E for moe_expert_ffn's workspace size)
size_t ffn_workspace_bytes(long long A, int F, int G) {
  // intermediate, then the fused kernel's per-block counters
  return ffn_inter_bytes(A, F) + (size_t)ffn_blocks_bound(A, G) * 4 + 1024;
}

}  // namespace

struct moe_stats {
  int L, E, s, device;
  void* block;                       // one allocation for everything below
  size_t block_bytes;
  uint32_t* ring_h;                  // [L][s][E]
  unsigned long long* hsum;          // [L][E]
  uint32_t* ring_c;                  // [L-1][s][E][E]
  unsigned long long* csum;          // [L-1][E][E]
  uint32_t* acc;                     // [E + E*E] (zero between calls)
  uint32_t* seg;                     // [front::kSegSlots][E] (zero between calls)
  uint32_t* ticket;                  // [2]: the ticket, then the one-launch front's arrival count
  double* dscratch;                  // [E + E*E] decay-weighted sums (moe_predict_decay), not exported
  size_t state_bytes;                // exported bytes (rings + sums), without header
};

namespace {
constexpr uint32_t kStatsMagic = 0x53454F4Du;  // "MOES"
struct StatsHeader {
  uint32_t magic, version;
  int32_t L, E, s, pad;
  uint64_t bytes;
};
}  // namespace

extern "C" {

const char* moe_version(void) { return MOE_VERSION_STRING; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_DEVICE: return "invalid device data";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

size_t moe_workspace_bytes(int op, int T, int k, int E, int H, int F) {
  if (T < 0 || k < 1 || k > 8 || E < 1 || E > 256) return 0;
  const long long A = (long long)T * k;
  if (op == MOE_OP_DISPATCH) return dispatch::workspace_bytes(A, E);
  if (op == MOE_OP_LAYER_FRONT) return front::workspace_bytes(T, E);
  if (op == MOE_OP_EXPERT_FFN) {
    if (F < 64 || F % 64 || H < 64 || H % 64) return 0;
    return ffn_workspace_bytes(A, F, 2 * E);
  }
  if (op == MOE_OP_EXPERT_FFN_COMBINE) {
    if (F < 64 || F % 64 || H < 64 || H % 64) return 0;
    return ((ffn_workspace_bytes(A, F, 2 * E) + 255) & ~(size_t)255) + (size_t)T * H * 4;
  }
  return 0;
}

// ------------------------------------------------------------------ stats
moe_status moe_stats_create(moe_stats** out, int L, int E, int window, void* stream) {
  if (!out) return fail(MOE_ERR_INVALID, "moe_stats_create: null handle pointer");
  *out = nullptr;
  if (L < 1 || L > 1024 || E < 1 || E > 256 || window < 1 || window > 1024)
    return fail(MOE_ERR_INVALID, "moe_stats_create: need 1<=L<=1024, 1<=E<=256, 1<=window<=1024");
  moe_stats* st = new (std::nothrow) moe_stats();
  if (!st) return fail(MOE_ERR_CUDA, "moe_stats_create: host allocation failed");
  st->L = L;
  st->E = E;
  st->s = window;
  cudaGetDevice(&st->device);
  const size_t nh = (size_t)L * window * E;
  const size_t nhs = (size_t)L * E;
  const size_t nc = (size_t)(L - 1) * window * E * E;
  const size_t ncs = (size_t)(L - 1) * E * E;
  const size_t nacc = (size_t)E + (size_t)E * E;
  const size_t nseg = (size_t)front::kSegSlots * E;
  // layout: 8-byte sums first, then 4-byte arrays, then the fp64 scratch
  const size_t four = ((nh + nc + nacc + nseg + 2) * 4 + 7) / 8 * 8;
  const size_t bytes = (nhs + ncs) * 8 + four + nacc * 8;
  cudaError_t e = cudaMalloc(&st->block, bytes);
  if (e != cudaSuccess) {
    delete st;
    return cuda_status(e, "moe_stats_create: cudaMalloc");
  }
  st->block_bytes = bytes;
  char* p = static_cast<char*>(st->block);
  st->hsum = reinterpret_cast<unsigned long long*>(p);
  p += nhs * 8;
  st->csum = reinterpret_cast<unsigned long long*>(p);
  p += ncs * 8;
  st->ring_h = reinterpret_cast<uint32_t*>(p);
  p += nh * 4;
  st->ring_c = reinterpret_cast<uint32_t*>(p);
  p += nc * 4;
  st->acc = reinterpret_cast<uint32_t*>(p);
  p += nacc * 4;
  st->seg = reinterpret_cast<uint32_t*>(p);
  p += nseg * 4;
  st->ticket = reinterpret_cast<uint32_t*>(p);
  st->dscratch = reinterpret_cast<double*>(static_cast<char*>(st->block) + (nhs + ncs) * 8 + four);
  st->state_bytes = (nhs + ncs) * 8 + (nh + nc) * 4;
  e = cudaMemsetAsync(st->block, 0, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaFree(st->block);
    delete st;
    return cuda_status(e, "moe_stats_create: cudaMemsetAsync");
  }
  *out = st;
  return MOE_OK;
}

moe_status moe_stats_destroy(moe_stats* st) {
  if (!st) return MOE_OK;
  cudaError_t e = cudaFree(st->block);
  delete st;
  return cuda_status(e, "moe_stats_destroy: cudaFree");
}

size_t moe_stats_bytes(const moe_stats* st) { return st ? sizeof(StatsHeader) + st->state_bytes : 0; }

moe_status moe_stats_export(const moe_stats* st, void* host_buf, size_t bytes) {
  if (!st || !host_buf) return fail(MOE_ERR_INVALID, "moe_stats_export: null argument");
  if (bytes < moe_stats_bytes(st)) return fail(MOE_ERR_INVALID, "moe_stats_export: buffer too small");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e, "moe_stats_export: sync");
  StatsHeader h{kStatsMagic, 1u, st->L, st->E, st->s, 0, (uint64_t)st->state_bytes};
  memcpy(host_buf, &h, sizeof(h));
  e = cudaMemcpy(static_cast<char*>(host_buf) + sizeof(h), st->block, st->state_bytes, cudaMemcpyDeviceToHost);
  return cuda_status(e, "moe_stats_export: cudaMemcpy");
}

moe_status moe_stats_import(moe_stats* st, const void* host_buf, size_t bytes) {
  if (!st || !host_buf) return fail(MOE_ERR_INVALID, "moe_stats_import: null argument");
  if (bytes < moe_stats_bytes(st)) return fail(MOE_ERR_INVALID, "moe_stats_import: buffer too small");
  StatsHeader h;
  memcpy(&h, host_buf, sizeof(h));
  if (h.magic != kStatsMagic || h.version != 1u || h.L != st->L || h.E != st->E || h.s != st->s ||
      h.bytes != st->state_bytes)
    return fail(MOE_ERR_INVALID, "moe_stats_import: buffer does not match this handle (L, E, window)");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e, "moe_stats_import: sync");
  e = cudaMemcpy(st->block, static_cast<const char*>(host_buf) + sizeof(h), st->state_bytes, cudaMemcpyHostToDevice);
  return cuda_status(e, "moe_stats_import: cudaMemcpy");
}

// ------------------------------------------------------------------ route
moe_status moe_route(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w, void* stream) {
  if (T < 0 || E < 1 || E > 256 || k < 1 || k > 8 || k > E)
    return fail(MOE_ERR_INVALID, "moe_route: need T>=0, 1<=E<=256, 1<=k<=min(E,8)");
  if ((long long)T * k >= (1LL << 31)) return fail(MOE_ERR_INVALID, "moe_route: T*k too large");
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w) return fail(MOE_ERR_INVALID, "moe_route: null pointer");
  if (!aligned(logits, 16) || !aligned(idx, 4) || !aligned(w, 4))
    return fail(MOE_ERR_INVALID, "moe_route: logits must be 16-byte aligned, idx/w 4-byte aligned");
  return cuda_status(route::launch(logits, T, E, k, renorm ? 1 : 0, idx, w, static_cast<cudaStream_t>(stream)),
                     "moe_route launch");
}

// ------------------------------------------------------------------ stats update / predict
moe_status moe_stats_update(moe_stats* st, int64_t iter, int layer, const int32_t* idx_layer,
                            const int32_t* idx_prev, int T, int k, int32_t* hist_out, void* stream) {
  if (!st) return fail(MOE_ERR_INVALID, "moe_stats_update: null handle");
  if (iter < 0 || layer < 0 || layer >= st->L || T < 0 || k < 1 || k > 8 || k > st->E)
    return fail(MOE_ERR_INVALID, "moe_stats_update: bad iter/layer/T/k");
  if ((long long)T * k >= (1LL << 31)) return fail(MOE_ERR_INVALID, "moe_stats_update: T*k too large");
  if (T > 0 && !idx_layer) return fail(MOE_ERR_INVALID, "moe_stats_update: null idx_layer");
  if (layer > 0 && T > 0 && !idx_prev) return fail(MOE_ERR_INVALID, "moe_stats_update: layer > 0 needs idx_prev");
  if (layer == 0 && idx_prev) return fail(MOE_ERR_INVALID, "moe_stats_update: idx_prev must be NULL for layer 0");
  DeviceInfo* d = nullptr;
  moe_status ms = device_info(&d);
  if (ms != MOE_OK) return ms;
  const int E = st->E, s = st->s;
  const int slot = (int)(iter % s);
  stats::UpdateArgs a;
  a.idx_cur = idx_layer;
  a.idx_prev = layer > 0 ? idx_prev : nullptr;
  a.has_prev = layer > 0 ? 1 : 0;
  a.T = T;
  a.k = k;
  a.E = E;
  a.acc_h = st->acc;
  a.acc_c = st->acc + E;
  a.ticket = st->ticket;
  a.ring_h = st->ring_h + ((size_t)layer * s + slot) * E;
  a.hsum = st->hsum + (size_t)layer * E;
  a.ring_c = layer > 0 ? st->ring_c + ((size_t)(layer - 1) * s + slot) * E * E : nullptr;
  a.csum = layer > 0 ? st->csum + (size_t)(layer - 1) * E * E : nullptr;
  a.hist_out = hist_out;
  return cuda_status(stats::launch_update(a, d->num_sms, static_cast<cudaStream_t>(stream)),
                     "moe_stats_update launch");
}

moe_status moe_predict(moe_stats* st, int layer, float* p_seq, float* cond, float* p_next, void* stream) {
  if (!st) return fail(MOE_ERR_INVALID, "moe_predict: null handle");
  if (layer < 0 || layer >= st->L) return fail(MOE_ERR_INVALID, "moe_predict: layer out of range");
  if (!p_seq) return fail(MOE_ERR_INVALID, "moe_predict: null p_seq");
  if (layer == st->L - 1 && (cond || p_next))
    return fail(MOE_ERR_INVALID, "moe_predict: the last layer has no next layer (cond/p_next must be NULL)");
  const int E = st->E;
  const unsigned long long* csum = (layer < st->L - 1) ? st->csum + (size_t)layer * E * E : nullptr;
  stats::predict_kernel<<<1, stats::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      st->hsum + (size_t)layer * E, csum, E, p_seq, cond, p_next);
  return cuda_status(cudaGetLastError(), "moe_predict launch");
}

moe_status moe_predict_decay(moe_stats* st, int layer, int64_t iter, double lambda, float* p_seq, float* cond,
                             float* p_next, void* stream) {
  if (!st) return fail(MOE_ERR_INVALID, "moe_predict_decay: null handle");
  if (layer < 0 || layer >= st->L) return fail(MOE_ERR_INVALID, "moe_predict_decay: layer out of range");
  if (iter < 0) return fail(MOE_ERR_INVALID, "moe_predict_decay: iter must be >= 0");
  if (!(lambda >= 0.0 && lambda <= 1.0)) return fail(MOE_ERR_INVALID, "moe_predict_decay: lambda must lie in [0, 1]");
  if (!p_seq) return fail(MOE_ERR_INVALID, "moe_predict_decay: null p_seq");
  if (layer == st->L - 1 && (cond || p_next))
    return fail(MOE_ERR_INVALID, "moe_predict_decay: the last layer has no next layer (cond/p_next must be NULL)");
  const int E = st->E, s = st->s;
  const uint32_t* rh = st->ring_h + (size_t)layer * s * E;
  const uint32_t* rc = (layer < st->L - 1) ? st->ring_c + (size_t)layer * s * E * E : nullptr;
  stats::predict_decay_kernel<<<1, stats::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      rh, rc, E, s, (long long)iter, lambda, st->dscratch, p_seq, cond, p_next);
  return cuda_status(cudaGetLastError(), "moe_predict_decay launch");
}

// ------------------------------------------------------------------ replicate
moe_status moe_replicate(const int32_t* load, int E, int64_t total, int thresh_num, int thresh_den, int max_copies,
                         int32_t* copies, int32_t* rep_base, int32_t* group_expert, void* stream) {
  if (E < 1 || E > 256 || total < 0 || total >= (1LL << 31))
    return fail(MOE_ERR_INVALID, "moe_replicate: need 1<=E<=256, 0<=total<2^31");
  if (thresh_num < 1 || thresh_den < 1 || thresh_num > 1024 || thresh_den > 1024)
    return fail(MOE_ERR_INVALID, "moe_replicate: threshold num/den must be in [1, 1024]");
  if (max_copies < -1) return fail(MOE_ERR_INVALID, "moe_replicate: max_copies must be >= -1");
  if (!load || !copies || !rep_base || !group_expert) return fail(MOE_ERR_INVALID, "moe_replicate: null pointer");
  return cuda_status(replicate::launch(load, E, total, thresh_num, thresh_den, max_copies, copies, rep_base,
                                       group_expert, static_cast<cudaStream_t>(stream)),
                     "moe_replicate launch");
}

moe_status moe_replicate_predicted(const float* p_next, int E, int64_t total, int thresh_num, int thresh_den,
                                   int max_copies, int budget, int32_t* load_out, int32_t* copies, int32_t* rep_base,
                                   int32_t* group_expert, void* stream) {
  if (E < 1 || E > 256) return fail(MOE_ERR_INVALID, "moe_replicate_predicted: need 1<=E<=256");
  if (total < 1 || total >= (1LL << 29))
    return fail(MOE_ERR_INVALID, "moe_replicate_predicted: need 1 <= total < 2^29 (exact quotas)");
  if (thresh_num < 1 || thresh_den < 1 || thresh_num > 1024 || thresh_den > 1024)
    return fail(MOE_ERR_INVALID, "moe_replicate_predicted: threshold num/den must be in [1, 1024]");
  if (max_copies < -1 || budget < -1)
    return fail(MOE_ERR_INVALID, "moe_replicate_predicted: max_copies and budget must be >= -1");
  if (!p_next || !load_out || !copies || !rep_base || !group_expert)
    return fail(MOE_ERR_INVALID, "moe_replicate_predicted: null pointer");
  return cuda_status(replicate::launch_predicted(p_next, E, total, thresh_num, thresh_den, max_copies, budget,
                                                 load_out, copies, rep_base, group_expert,
                                                 static_cast<cudaStream_t>(stream)),
                     "moe_replicate_predicted launch");
}

// ------------------------------------------------------------------ dispatch
moe_status moe_dispatch(const uint16_t* x, const int32_t* idx, int T, int k, int H, int E, const int32_t* rep_base,
                        int32_t* group_offsets, int32_t* perm, int32_t* inv_perm, uint16_t* xp, void* workspace,
                        size_t ws_bytes, void* stream) {
  if (T < 0 || E < 1 || E > 256 || k < 1 || k > 8 || k > E || H < 8 || H % 8)
    return fail(MOE_ERR_INVALID, "moe_dispatch: need T>=0, 1<=E<=256, 1<=k<=min(E,8), H a positive multiple of 8");
  if ((long long)T * k >= (1LL << 31)) return fail(MOE_ERR_INVALID, "moe_dispatch: T*k too large");
  if (!group_offsets) return fail(MOE_ERR_INVALID, "moe_dispatch: null group_offsets");
  if ((x == nullptr) != (xp == nullptr)) return fail(MOE_ERR_INVALID, "moe_dispatch: x and xp must both be set or both NULL");
  if (T > 0 && (!idx || !perm || !inv_perm || !workspace)) return fail(MOE_ERR_INVALID, "moe_dispatch: null pointer");
  if (x && (!aligned(x, 16) || !aligned(xp, 16))) return fail(MOE_ERR_INVALID, "moe_dispatch: x/xp must be 16-byte aligned");
  if (workspace && !aligned(workspace, 16)) return fail(MOE_ERR_INVALID, "moe_dispatch: workspace must be 16-byte aligned");
  if (T > 0 && ws_bytes < dispatch::workspace_bytes((long long)T * k, E))
    return fail(MOE_ERR_WORKSPACE, "moe_dispatch: workspace needs %zu bytes", dispatch::workspace_bytes((long long)T * k, E));
  DeviceInfo* d = nullptr;
  moe_status ms = device_info(&d);
  if (ms != MOE_OK) return ms;
  dispatch::Args a{x, idx, (long long)T, k, H, E, rep_base, group_offsets, perm, inv_perm, xp, workspace};
  return cuda_status(dispatch::launch(a, d->num_sms, static_cast<cudaStream_t>(stream)), "moe_dispatch launch");
}

// ------------------------------------------------------------------ fused front
moe_status moe_layer_front(const float* logits, const uint16_t* x, int T, int E, int k, int H, int renorm,
                           moe_stats* st, int64_t iter, int layer, const int32_t* idx_prev, int replicate,
                           int thresh_num, int thresh_den, int max_copies, const float* rep_share, int budget,
                           int32_t* idx, float* w,
                           int32_t* hist_out, float* p_seq, float* cond, float* p_next, int32_t* copies,
                           int32_t* rep_base, int32_t* group_expert, int32_t* group_offsets, int32_t* perm,
                           int32_t* inv_perm, uint16_t* xp, void* workspace, size_t ws_bytes, void* stream) {
  if (!st) return fail(MOE_ERR_INVALID, "moe_layer_front: null stats handle");
  if (E != st->E) return fail(MOE_ERR_INVALID, "moe_layer_front: E differs from the stats handle's");
  if (T < 0 || k < 1 || k > 8 || k > E || H < 8 || H % 8)
    return fail(MOE_ERR_INVALID, "moe_layer_front: need T>=0, 1<=k<=min(E,8), H a positive multiple of 8");
  if ((long long)T * k >= (1LL << 31)) return fail(MOE_ERR_INVALID, "moe_layer_front: T*k too large");
  if (iter < 0 || layer < 0 || layer >= st->L) return fail(MOE_ERR_INVALID, "moe_layer_front: bad iter/layer");
  if (layer > 0 && T > 0 && !idx_prev) return fail(MOE_ERR_INVALID, "moe_layer_front: layer > 0 needs idx_prev");
  if (layer == 0 && idx_prev) return fail(MOE_ERR_INVALID, "moe_layer_front: idx_prev must be NULL for layer 0");
  if (layer == st->L - 1 && (cond || p_next))
    return fail(MOE_ERR_INVALID, "moe_layer_front: the last layer has no next layer (cond/p_next must be NULL)");
  if (!p_seq && (cond || p_next)) return fail(MOE_ERR_INVALID, "moe_layer_front: cond/p_next need p_seq");
  if (replicate && (!copies || !rep_base || !group_expert))
    return fail(MOE_ERR_INVALID, "moe_layer_front: replication needs copies, rep_base, group_expert");
  if (replicate && (thresh_num < 1 || thresh_den < 1 || thresh_num > 1024 || thresh_den > 1024 || max_copies < -1 ||
                    budget < -1))
    return fail(MOE_ERR_INVALID, "moe_layer_front: bad replication threshold, cap or budget");
  if (replicate && rep_share && (long long)T * k >= (1LL << 29))
    return fail(MOE_ERR_INVALID, "moe_layer_front: replication from shares needs T*k < 2^29");
  if (!group_offsets) return fail(MOE_ERR_INVALID, "moe_layer_front: null group_offsets");
  if ((x == nullptr) != (xp == nullptr))
    return fail(MOE_ERR_INVALID, "moe_layer_front: x and xp must both be set or both NULL");
  if (T == 0) {
    // empty batch: the separate calls handle it (window slot cleared, empty layout)
    moe_status r = moe_stats_update(st, iter, layer, nullptr, nullptr, 0, k, hist_out, stream);
    if (r != MOE_OK) return r;
    if (p_seq && (r = moe_predict(st, layer, p_seq, cond, p_next, stream)) != MOE_OK) return r;
    if (replicate) {
      if (!hist_out) return fail(MOE_ERR_INVALID, "moe_layer_front: an empty batch with replication needs hist_out");
      if ((r = moe_replicate(hist_out, E, 0, thresh_num, thresh_den, max_copies, copies, rep_base, group_expert,
                             stream)) != MOE_OK)
        return r;
    }
    return moe_dispatch(nullptr, nullptr, 0, k, H, E, nullptr, group_offsets, nullptr, nullptr, nullptr, nullptr, 0,
                        stream);
  }
  if (!logits || !idx || !w || !perm || !inv_perm || !workspace)
    return fail(MOE_ERR_INVALID, "moe_layer_front: null pointer");
  if (!aligned(logits, 16) || !aligned(workspace, 16) || (x && (!aligned(x, 16) || !aligned(xp, 16))))
    return fail(MOE_ERR_INVALID, "moe_layer_front: logits, workspace, x and xp must be 16-byte aligned");
  if (ws_bytes < front::workspace_bytes(T, E))
    return fail(MOE_ERR_WORKSPACE, "moe_layer_front: workspace needs %zu bytes", front::workspace_bytes(T, E));
  const int s = st->s;
  const int slot = (int)(iter % s);
  front::Args a{};
  a.logits = logits;
  a.T = T;
  a.E = E;
  a.k = k;
  a.renorm = renorm ? 1 : 0;
  a.idx = idx;
  a.w = w;
  a.has_prev = layer > 0 ? 1 : 0;
  a.idx_prev = idx_prev;
  a.acc_h = st->acc;
  a.acc_c = st->acc + E;
  a.seg_tot = st->seg;
  a.ticket = st->ticket;
  a.arrive = st->ticket + 1;
  a.ring_h = st->ring_h + ((size_t)layer * s + slot) * E;
  a.hsum = st->hsum + (size_t)layer * E;
  a.ring_c = layer > 0 ? st->ring_c + ((size_t)(layer - 1) * s + slot) * E * E : nullptr;
  a.csum = layer > 0 ? st->csum + (size_t)(layer - 1) * E * E : nullptr;
  a.hist_out = hist_out;
  a.pred_csum = (layer < st->L - 1) ? st->csum + (size_t)layer * E * E : nullptr;
  a.p_seq = p_seq;
  a.cond = cond;
  a.p_next = p_next;
  a.replicate = replicate ? 1 : 0;
  a.rep_share = replicate ? rep_share : nullptr;
  a.budget = budget;
  a.num = thresh_num;
  a.den = thresh_den;
  a.max_copies = max_copies;
  a.copies = copies;
  a.rep_base = rep_base;
  a.group_expert = group_expert;
  a.TT = front::tile_tokens(T);
  a.ntiles = front::num_tiles(T);
  a.counts = static_cast<int32_t*>(workspace);
  a.blk_tot = a.counts + a.ntiles * E;
  a.group_offsets = group_offsets;
  DeviceInfo* dinfo = nullptr;
  if (moe_status ds = device_info(&dinfo); ds != MOE_OK) return ds;
  return cuda_status(front::launch(a, x, H, xp, perm, inv_perm, dinfo->num_sms, static_cast<cudaStream_t>(stream)),
                     "moe_layer_front launch");
}

// ------------------------------------------------------------------ expert FFN
namespace {

// Kernel choice of the expert FFN (see moe_set_option): the CTA-pair kernels
// when the experts average >= 256 rows; among them the fused one (both GEMMs
// in one launch, tiles block by block) for experts of at most 16 MB of
// weights -- it re-reads larger experts' weights from DRAM per 256-row block
// (measured: +6% at 8 MB per expert, -12..-15% at 235-400 MB), where the
// two-launch kernel's order reuses each weight slice across blocks -- and
// never with gathered rows.  Depends only on the sizes and the options.
void ffn_choice(long long A, int E, int H, int F, int act, bool gather, bool* use_pair, bool* use_fused) {
  const int opt = g_opt_ffn_kernel.load(std::memory_order_relaxed);
  bool pair = A >= 256LL * E;
  if (opt == MOE_FFN_KERNEL_SINGLE) pair = false;
  if (opt == MOE_FFN_KERNEL_PAIR || opt == MOE_FFN_KERNEL_FUSED) pair = true;
  const long long expert_weight_bytes = (long long)(act == MOE_ACT_SWIGLU ? 3 : 2) * H * F * 2;
  *use_pair = pair;
  *use_fused = pair && !gather &&
               (opt == MOE_FFN_KERNEL_FUSED || (opt == MOE_FFN_KERNEL_AUTO && expert_weight_bytes <= (16LL << 20)));
}

// The combine fused into GEMM2 (moe_expert_ffn_combine): GEMM2's epilogues
// add w[perm[i]] * Y[i] into acc [T, H] fp32 (zeroed first), then one pass
// rounds acc to bf16 into out.
struct CombineArgs {
  const int32_t* perm;
  const float* w;
  int k;
  long long T;
  float* acc;
  uint16_t* out;
};

// The FFN entry points.  a_src == null: A (GEMM1's input rows) is `a`
// itself, [A, H] in dispatched order.  Otherwise `a` is x [T, H] and row i
// of A is x[a_src[i] / k], gathered by GEMM1's loads.  comb != null: the
// combine runs in GEMM2's epilogue instead of storing Y (y unused).
moe_status expert_ffn(const char* who, const uint16_t* a, const int32_t* a_src, int k, int T,
                      const int32_t* group_offsets, const int32_t* group_expert, int G, const int32_t* rep_base, int E,
                      int A,
                      const uint16_t* w1, const uint16_t* w3, const uint16_t* w2, int H, int F, moe_act act,
                      int small_group_threshold, uint16_t* y, void* workspace, size_t ws_bytes, void* stream,
                      const CombineArgs* comb = nullptr) {
  const uint16_t* xp = a;
  const bool gather = a_src != nullptr;
  if (E < 1 || E > ffn::MAX_G || A < 0) return fail(MOE_ERR_INVALID, "%s: need 1<=E<=%d, A>=0", who, ffn::MAX_G);
  if (G < 1 || G > ffn::MAX_G) return fail(MOE_ERR_INVALID, "%s: need 1 <= groups <= %d", who, ffn::MAX_G);
  if (H < 64 || H % 64 || F < 64 || F % 64) return fail(MOE_ERR_INVALID, "%s: H and F must be positive multiples of 64", who);
  if (act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID, "%s: unknown activation", who);
  if (small_group_threshold < 0) return fail(MOE_ERR_INVALID, "%s: small_group_threshold must be >= 0", who);
  if ((long long)E * H >= (1LL << 31) || (long long)E * F >= (1LL << 31))
    return fail(MOE_ERR_INVALID, "%s: weights too large", who);
  if (A == 0) return MOE_OK;
  if (!xp || !group_offsets || !w1 || !w2 || (!y && !comb) || !workspace)
    return fail(MOE_ERR_INVALID, "%s: null pointer", who);
  if (act == MOE_ACT_SWIGLU && !w3) return fail(MOE_ERR_INVALID, "%s: SwiGLU needs w3", who);
  if (!aligned(xp, 16) || !aligned(w1, 16) || !aligned(w2, 16) || (y && !aligned(y, 16)) || (w3 && !aligned(w3, 16)))
    return fail(MOE_ERR_INVALID, "%s: matrices must be 16-byte aligned", who);
  if (!aligned(workspace, 16)) return fail(MOE_ERR_INVALID, "%s: workspace must be 16-byte aligned", who);
  if (ws_bytes < ffn_workspace_bytes(A, F, G))
    return fail(MOE_ERR_WORKSPACE, "%s: workspace needs %zu bytes", who, ffn_workspace_bytes(A, F, G));
  const long long tiles_bound = ((long long)(A + ffn::BM - 1) / ffn::BM + G) *
                                (long long)((F + 63) / 64 + (H + 63) / 64);
  if (tiles_bound >= (1LL << 31)) return fail(MOE_ERR_INVALID, "%s: problem too large", who);

  DeviceInfo* d = nullptr;
  moe_status ms = device_info(&d);
  if (ms != MOE_OK) return ms;
  ms = get_encoder();
  if (ms != MOE_OK) return ms;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t* inter = static_cast<uint16_t*>(workspace);

  CUtensorMap mA1, mW1, mW3, mA2, mW2;
  // gathered rows: a one-row box, four rows per copy (tile::gather4)
  if ((ms = gather ? encode_2d(&mA1, xp, H, T, 64, 1) : encode_2d(&mA1, xp, H, A, 64, ffn::BM)) != MOE_OK) return ms;
  if ((ms = encode_2d(&mW1, w1, F, (uint64_t)E * H, 64, 64)) != MOE_OK) return ms;
  if (act == MOE_ACT_SWIGLU) {
    if ((ms = encode_2d(&mW3, w3, F, (uint64_t)E * H, 64, 64)) != MOE_OK) return ms;
  } else {
    mW3 = mW1;
  }
  if ((ms = encode_2d(&mA2, inter, F, A, 64, ffn::BM)) != MOE_OK) return ms;
  if ((ms = encode_2d(&mW2, w2, H, (uint64_t)E * F, 64, 64)) != MOE_OK) return ms;

  const int epi1 = act == MOE_ACT_SWIGLU ? ffn::kSwiglu : ffn::kGelu;
  // Kernel choice: the CTA-pair kernel works in 256-row pair tiles, so it is
  // used when the experts average at least 256 rows; the choice depends on
  // (A, E) only, so a call with and without replica groups takes the same path.
  bool use_pair = false, use_fused = false;
  ffn_choice(A, E, H, F, act, gather, &use_pair, &use_fused);
  if (comb) use_fused = false;  // the fused kernel's GEMM2 stores Y

  ffn::Params p1{};
  p1.group_offsets = group_offsets;
  p1.group_expert = group_expert;
  p1.G = G;
  p1.E = E;
  p1.A_rows = A;
  p1.K = H;
  p1.N_out = F;
  p1.out = inter;
  p1.flags = g_opt_ffn_selftest.exchange(0) ? 1 : 0;
  p1.rep_base = rep_base;
  p1.small_threshold = small_group_threshold;
  // SM split between the small-batch and the grouped kernels (every kernel
  // of the call gets the same split fields, so they agree on it); with the
  // option at 0 the grouped kernels take every expert and the small-batch
  // kernels are not launched
  const int small_sms_opt = g_opt_ffn_small_sms.load(std::memory_order_relaxed);
  if (small_group_threshold > 0) {
    p1.split_ctas = d->num_sms;
    p1.split_force = small_sms_opt;
    p1.split_pair = use_pair ? 1 : 0;
    p1.split_rows = use_pair ? ffn2::BMP : ffn::BM;
    p1.ffn_H = H;
    p1.ffn_F = F;
    p1.ffn_mats = act == MOE_ACT_SWIGLU ? 3 : 2;
  }
  p1.a_src = a_src;
  p1.a_src_div = gather ? k : 1;
  p1.a_src_rows = gather ? T : 0;
  ffn::Params p2 = p1;
  p2.flags = 0;
  p2.a_src = nullptr;
  p2.a_src_div = 1;
  p2.a_src_rows = 0;
  p2.K = F;
  p2.N_out = H;
  p2.out = y;
  if (comb) {
    p2.comb_perm = comb->perm;
    p2.comb_w = comb->w;
    p2.comb_k = comb->k;
    p2.comb_acc = comb->acc;
  }
  const int epi2 = comb ? ffn::kCombine : ffn::kStore;

  // small-batch kernels (experts with fewer than small_group_threshold rows)
  CUtensorMap mS1, mS2;
  ffn::Params ps1 = p1, ps2 = p2;
  ps1.flags = 0;
  ps1.n_tiles = (F + ffn_small::BMF - 1) / ffn_small::BMF;
  ps2.n_tiles = (H + ffn_small::BMF - 1) / ffn_small::BMF;
  const bool small_path = small_group_threshold > 0 && small_sms_opt != 0;
  if (small_path) {
    if (gather)
      mS1 = mA1;
    else if ((ms = encode_2d(&mS1, xp, H, A, 64, ffn_small::BT)) != MOE_OK)
      return ms;
    if ((ms = encode_2d(&mS2, inter, F, A, 64, ffn_small::BT)) != MOE_OK) return ms;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < 4; ++i) {
      if (d->small_attr[i]) continue;
      const void* fn = i == 0 ? (const void*)ffn_small::small_kernel<ffn::kGelu>
                     : i == 1 ? (const void*)ffn_small::small_kernel<ffn::kSwiglu>
                     : i == 2 ? (const void*)ffn_small::small_kernel<ffn::kStore>
                              : (const void*)ffn_small::small_kernel<ffn::kCombine>;
      const int bytes = i == 0 ? (int)ffn_small::smem_bytes<ffn::kGelu>()
                      : i == 1 ? (int)ffn_small::smem_bytes<ffn::kSwiglu>()
                      : i == 2 ? (int)ffn_small::smem_bytes<ffn::kStore>()
                               : (int)ffn_small::smem_bytes<ffn::kCombine>();
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e != cudaSuccess) return cuda_at(who, e, "cudaFuncSetAttribute (small)");
      d->small_attr[i] = true;
    }
  }
  const long long small_bound = (long long)G + (long long)A / ffn_small::BT + 1;
  auto small_grid = [&](const ffn::Params& p) {
    long long g = small_bound * p.n_tiles;
    if (g > d->num_sms) g = d->num_sms;
    return (unsigned)(g < 1 ? 1 : g);
  };
  // The small-batch kernels touch other rows of inter and y than the grouped
  // kernels (experts below the threshold), so they form a second chain,
  // small1 -> small2, on the device's side stream: forked from `st` before
  // GEMM1 and joined back after GEMM2 (the whole sequence is enqueued under
  // one lock, so concurrent callers cannot interleave their forks and joins).
  auto launch_small_chain = [&](cudaStream_t ss) -> cudaError_t {
    if (epi1 == ffn::kSwiglu)
      ffn_small::small_kernel<ffn::kSwiglu><<<small_grid(ps1), ffn_small::THREADS,
                                              ffn_small::smem_bytes<ffn::kSwiglu>(), ss>>>(mS1, mW1, mW3, ps1);
    else
      ffn_small::small_kernel<ffn::kGelu><<<small_grid(ps1), ffn_small::THREADS, ffn_small::smem_bytes<ffn::kGelu>(),
                                            ss>>>(mS1, mW1, mW3, ps1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (epi2 == ffn::kCombine)
      ffn_small::small_kernel<ffn::kCombine><<<small_grid(ps2), ffn_small::THREADS,
                                               ffn_small::smem_bytes<ffn::kCombine>(), ss>>>(mS2, mW2, mW2, ps2);
    else
      ffn_small::small_kernel<ffn::kStore><<<small_grid(ps2), ffn_small::THREADS, ffn_small::smem_bytes<ffn::kStore>(),
                                             ss>>>(mS2, mW2, mW2, ps2);
    return cudaGetLastError();
  };
  std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);
  // forks the side chain off `st`, right before the first grouped kernel
  // (the combine accumulator is zeroed first, before either chain adds to it)
  auto fork = [&]() -> cudaError_t {
    if (comb) {
      cudaError_t z = cudaMemsetAsync(comb->acc, 0, (size_t)comb->T * H * sizeof(float), st);
      if (z != cudaSuccess) return z;
    }
    if (!small_path) return cudaSuccess;
    side_lock.lock();
    cudaError_t e = cudaEventRecord(d->fork_ev, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->side, d->fork_ev, 0);
    if (e != cudaSuccess) side_lock.unlock();
    return e;
  };
  // joins the side chain back into `st` (after the grouped kernels are enqueued)
  auto finish = [&](cudaError_t e_main, const char* what) -> moe_status {
    moe_status r;
    if (!small_path) {
      r = cuda_at(who, e_main, what);
    } else {
      cudaError_t e = launch_small_chain(d->side);
      cudaError_t j = cudaEventRecord(d->join_ev, d->side);
      if (j == cudaSuccess) j = cudaStreamWaitEvent(st, d->join_ev, 0);
      if (e_main != cudaSuccess) return cuda_at(who, e_main, what);
      if (e != cudaSuccess) return cuda_at(who, e, "small-batch kernels launch");
      r = cuda_at(who, j, "join of the small-batch chain");
    }
    if (r != MOE_OK || !comb) return r;
    return cuda_at(who, combine::launch_finalize(comb->acc, comb->T, H, comb->out, d->num_sms, st),
                   "combine finalize launch");
  };

  if (use_fused) {
    const int fi = epi1 == ffn::kSwiglu ? 1 : 0;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if (!d->fused_attr[fi]) {
        const void* fn = fi ? (const void*)ffn3::ffn_fused_kernel<ffn::kSwiglu>
                            : (const void*)ffn3::ffn_fused_kernel<ffn::kGelu>;
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ffn2::kSmemBytes);
        if (e != cudaSuccess) return cuda_at(who, e, "cudaFuncSetAttribute (fused)");
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (d->num_sms / 2), 1, 1);
        cfg.blockDim = dim3(ffn2::THREADS, 1, 1);
        cfg.dynamicSmemBytes = ffn2::kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
        if (e != cudaSuccess || n < 1)
          return cuda_at(who, e != cudaSuccess ? e : cudaErrorInvalidConfiguration,
                         "cudaOccupancyMaxActiveClusters (fused)");
        d->fused_clusters[fi] = n;
        d->fused_attr[fi] = true;
      }
    }
    // weight tiles: one 3-D box of both 64-column chunks of a CTA's half
    CUtensorMap mW1q, mW3q, mW2q;
    if ((ms = encode_w3d(&mW1q, w1, F, (uint64_t)E * H, 2)) != MOE_OK) return ms;
    if (act == MOE_ACT_SWIGLU) {
      if ((ms = encode_w3d(&mW3q, w3, F, (uint64_t)E * H, 2)) != MOE_OK) return ms;
    } else {
      mW3q = mW1q;
    }
    if ((ms = encode_w3d(&mW2q, w2, H, (uint64_t)E * F, 2)) != MOE_OK) return ms;
    ffn3::FusedParams fp;
    fp.p1 = p1;
    fp.p2 = p2;
    fp.p1.b3d = fp.p2.b3d = 1;
    fp.p1.n_tiles = act == MOE_ACT_SWIGLU ? (F + ffn2::BN / 2 - 1) / (ffn2::BN / 2) : (F + ffn2::BN - 1) / ffn2::BN;
    fp.p2.n_tiles = (H + ffn2::BN - 1) / ffn2::BN;
    const long long blocks = ffn_blocks_bound(A, G);
    fp.done = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + ffn_inter_bytes(A, F));
    const int npairs_max = d->fused_clusters[fi];
    const int per_block = fp.p1.n_tiles + fp.p2.n_tiles;
    // about three rounds of tiles between a block's GEMM1 and GEMM2 tiles
    // (measured on the moe_gpt_stream layer, FFN us: 1 round 260, 2 rounds
    // 228, 3 rounds 223.6, 4 rounds 223.8)
    fp.lag = (3 * npairs_max + per_block - 1) / per_block + 1;
    long long pairs = blocks * per_block;
    if (pairs > npairs_max) pairs = npairs_max;
    cudaError_t e = cudaMemsetAsync(fp.done, 0, (size_t)blocks * 4, st);
    if (e != cudaSuccess) return cuda_at(who, e, "cudaMemsetAsync (block counters)");
    if (cudaError_t fe = fork(); fe != cudaSuccess) return cuda_at(who, fe, "fork of the small-batch chain");
    cudaError_t le = launch_pdl(fi ? ffn3::ffn_fused_kernel<ffn::kSwiglu> : ffn3::ffn_fused_kernel<ffn::kGelu>,
                                dim3((unsigned)(2 * pairs)), dim3(ffn2::THREADS), ffn2::kSmemBytes, st, mA1, mW1q, mW3q,
                                mA2, mW2q, fp);
    return finish(le, "fused FFN launch");
  }

  if (use_pair) {
    {
      std::lock_guard<std::mutex> lk(g_mu);
      for (int i = 0; i < 4; ++i) {
        if (d->pair_attr[i]) continue;
        const void* fn = i == 0 ? (const void*)ffn2::gemm_pair_kernel<ffn::kGelu>
                       : i == 1 ? (const void*)ffn2::gemm_pair_kernel<ffn::kSwiglu>
                       : i == 2 ? (const void*)ffn2::gemm_pair_kernel<ffn::kStore>
                                : (const void*)ffn2::gemm_pair_kernel<ffn::kCombine>;
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ffn2::kSmemBytes);
        if (e != cudaSuccess) return cuda_at(who, e, "cudaFuncSetAttribute (pair)");
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (d->num_sms / 2), 1, 1);
        cfg.blockDim = dim3(ffn2::THREADS, 1, 1);
        cfg.dynamicSmemBytes = ffn2::kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
        if (e != cudaSuccess || n < 1) return cuda_at(who, e != cudaSuccess ? e : cudaErrorInvalidConfiguration,
                                                          "cudaOccupancyMaxActiveClusters");
        d->pair_clusters[i] = n;
        d->pair_attr[i] = true;
      }
    }
    p1.n_tiles = act == MOE_ACT_SWIGLU ? (F + ffn2::BN / 2 - 1) / (ffn2::BN / 2) : (F + ffn2::BN - 1) / ffn2::BN;
    p2.n_tiles = (H + ffn2::BN - 1) / ffn2::BN;
    CUtensorMap mW1q, mW3q, mW2q;
    if ((ms = encode_w3d(&mW1q, w1, F, (uint64_t)E * H, 2)) != MOE_OK) return ms;
    if (act == MOE_ACT_SWIGLU) {
      if ((ms = encode_w3d(&mW3q, w3, F, (uint64_t)E * H, 2)) != MOE_OK) return ms;
    } else {
      mW3q = mW1q;
    }
    if ((ms = encode_w3d(&mW2q, w2, H, (uint64_t)E * F, 2)) != MOE_OK) return ms;
    p1.b3d = p2.b3d = 1;
    const long long pt_bound = (long long)(A + ffn2::BMP - 1) / ffn2::BMP + G;
    auto grid_for = [&](const ffn::Params& p, int inst) {
      long long pairs = pt_bound * p.n_tiles;
      if (pairs > d->pair_clusters[inst]) pairs = d->pair_clusters[inst];
      return (unsigned)(2 * (pairs < 1 ? 1 : pairs));
    };
    if (cudaError_t fe = fork(); fe != cudaSuccess) return cuda_at(who, fe, "fork of the small-batch chain");
    cudaError_t e = launch_pdl(epi1 == ffn::kSwiglu ? ffn2::gemm_pair_kernel<ffn::kSwiglu>
                                                    : ffn2::gemm_pair_kernel<ffn::kGelu>,
                               dim3(grid_for(p1, epi1 == ffn::kSwiglu ? 1 : 0)), dim3(ffn2::THREADS),
                               ffn2::kSmemBytes, st, mA1, mW1q, mW3q, p1);
    if (e != cudaSuccess) return finish(e, "GEMM1 (pair) launch");
    e = launch_pdl(comb ? ffn2::gemm_pair_kernel<ffn::kCombine> : ffn2::gemm_pair_kernel<ffn::kStore>,
                   dim3(grid_for(p2, comb ? 3 : 2)), dim3(ffn2::THREADS), ffn2::kSmemBytes, st, mA2, mW2q, mW2q, p2);
    return finish(e, "GEMM2 (pair) launch");
  }

  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < 4; ++i) {
      if (d->ffn_attr[i]) continue;
      const void* fn = i == 0 ? (const void*)ffn::gemm_kernel<ffn::kGelu>
                     : i == 1 ? (const void*)ffn::gemm_kernel<ffn::kSwiglu>
                     : i == 2 ? (const void*)ffn::gemm_kernel<ffn::kStore>
                              : (const void*)ffn::gemm_kernel<ffn::kCombine>;
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ffn::kSmemBytes);
      if (e != cudaSuccess) return cuda_at(who, e, "cudaFuncSetAttribute");
      d->ffn_attr[i] = true;
    }
  }
  p1.n_tiles = act == MOE_ACT_SWIGLU ? (F + ffn::BN / 2 - 1) / (ffn::BN / 2) : (F + ffn::BN - 1) / ffn::BN;
  p2.n_tiles = (H + ffn::BN - 1) / ffn::BN;
  // weight tiles: one 3-D box per matrix and stage (four chunks, or two of
  // each of W1 and W3)
  CUtensorMap mW1q, mW3q, mW2q;
  if ((ms = encode_w3d(&mW1q, w1, F, (uint64_t)E * H, act == MOE_ACT_SWIGLU ? 2 : 4)) != MOE_OK) return ms;
  if (act == MOE_ACT_SWIGLU) {
    if ((ms = encode_w3d(&mW3q, w3, F, (uint64_t)E * H, 2)) != MOE_OK) return ms;
  } else {
    mW3q = mW1q;
  }
  if ((ms = encode_w3d(&mW2q, w2, H, (uint64_t)E * F, 4)) != MOE_OK) return ms;
  p1.b3d = p2.b3d = 1;
  const long long mt_bound = (long long)(A + ffn::BM - 1) / ffn::BM + G;
  auto grid_for = [&](const ffn::Params& p) {
    long long g = mt_bound * p.n_tiles;
    if (g > d->num_sms) g = d->num_sms;
    return (unsigned)(g < 1 ? 1 : g);
  };
  if (cudaError_t fe = fork(); fe != cudaSuccess) return cuda_at(who, fe, "fork of the small-batch chain");
  if (epi1 == ffn::kSwiglu)
    ffn::gemm_kernel<ffn::kSwiglu><<<grid_for(p1), ffn::THREADS, ffn::kSmemBytes, st>>>(mA1, mW1q, mW3q, p1);
  else
    ffn::gemm_kernel<ffn::kGelu><<<grid_for(p1), ffn::THREADS, ffn::kSmemBytes, st>>>(mA1, mW1q, mW3q, p1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return finish(e, "GEMM1 launch");
  if (comb)
    ffn::gemm_kernel<ffn::kCombine><<<grid_for(p2), ffn::THREADS, ffn::kSmemBytes, st>>>(mA2, mW2q, mW2q, p2);
  else
    ffn::gemm_kernel<ffn::kStore><<<grid_for(p2), ffn::THREADS, ffn::kSmemBytes, st>>>(mA2, mW2q, mW2q, p2);
  return finish(cudaGetLastError(), "GEMM2 launch");
}

}  // namespace

moe_status moe_expert_ffn(const uint16_t* xp, const int32_t* group_offsets, const int32_t* group_expert,
                          const int32_t* rep_base, int E, int A, const uint16_t* w1, const uint16_t* w3,
                          const uint16_t* w2, int H, int F, moe_act act, int small_group_threshold, uint16_t* y,
                          void* workspace, size_t ws_bytes, void* stream) {
  if (E < 1 || E > 256) return fail(MOE_ERR_INVALID, "moe_expert_ffn: need 1<=E<=256");
  return expert_ffn("moe_expert_ffn", xp, nullptr, 1, 0, group_offsets, group_expert, group_expert ? 2 * E : E,
                    rep_base, E, A, w1, w3, w2, H, F, act, small_group_threshold, y, workspace, ws_bytes, stream);
}

moe_status moe_expert_ffn_gather(const uint16_t* x, int T, const int32_t* perm, int k, const int32_t* group_offsets,
                                 const int32_t* group_expert, const int32_t* rep_base, int E, const uint16_t* w1,
                                 const uint16_t* w3, const uint16_t* w2, int H, int F, moe_act act,
                                 int small_group_threshold, uint16_t* y, void* workspace, size_t ws_bytes,
                                 void* stream) {
  if (T < 0 || k < 1 || k > 8 || k > E) return fail(MOE_ERR_INVALID, "moe_expert_ffn_gather: need T>=0, 1<=k<=min(E,8)");
  if ((long long)T * k >= (1LL << 31)) return fail(MOE_ERR_INVALID, "moe_expert_ffn_gather: T*k too large");
  if (T > 0 && (!x || !perm)) return fail(MOE_ERR_INVALID, "moe_expert_ffn_gather: null pointer");
  if (E < 1 || E > 256) return fail(MOE_ERR_INVALID, "moe_expert_ffn_gather: need 1<=E<=256");
  return expert_ffn("moe_expert_ffn_gather", x, T > 0 ? perm : nullptr, k, T, group_offsets, group_expert,
                    group_expert ? 2 * E : E, rep_base, E, T * k, w1, w3, w2, H, F, act, small_group_threshold, y,
                    workspace, ws_bytes, stream);
}

static size_t ffn_combine_acc_offset(long long A, int F, int G) { return (ffn_workspace_bytes(A, F, G) + 255) & ~(size_t)255; }

moe_status moe_expert_ffn_combine(const uint16_t* xp, const int32_t* group_offsets, const int32_t* group_expert,
                                  const int32_t* rep_base, int E, const int32_t* perm, const float* w, int T, int k,
                                  const uint16_t* w1, const uint16_t* w3, const uint16_t* w2, int H, int F,
                                  moe_act act, int small_group_threshold, uint16_t* out, void* workspace,
                                  size_t ws_bytes, void* stream) {
  const char* who = "moe_expert_ffn_combine";
  if (E < 1 || E > 256 || T < 0 || k < 1 || k > 8 || k > E)
    return fail(MOE_ERR_INVALID, "%s: need 1<=E<=256, T>=0, 1<=k<=min(E,8)", who);
  if ((long long)T * k >= (1LL << 31)) return fail(MOE_ERR_INVALID, "%s: T*k too large", who);
  if (H < 64 || H % 64 || F < 64 || F % 64) return fail(MOE_ERR_INVALID, "%s: H and F must be positive multiples of 64", who);
  if (T == 0) return MOE_OK;
  if (!perm || !w || !out || !workspace) return fail(MOE_ERR_INVALID, "%s: null pointer", who);
  if (!aligned(out, 16) || !aligned(workspace, 256))
    return fail(MOE_ERR_INVALID, "%s: out must be 16-byte aligned, the workspace 256-byte aligned", who);
  const int G = group_expert ? 2 * E : E;
  const long long A = (long long)T * k;
  const size_t off = ffn_combine_acc_offset(A, F, G);
  if (ws_bytes < off + (size_t)T * H * 4)
    return fail(MOE_ERR_WORKSPACE, "%s: workspace needs %zu bytes", who, off + (size_t)T * H * 4);
  CombineArgs cb{perm, w, k, T, reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + off), out};
  return expert_ffn(who, xp, nullptr, 1, 0, group_offsets, group_expert, G, rep_base, E, (int)A, w1, w3, w2, H, F,
                    act, small_group_threshold, nullptr, workspace, off, stream, &cb);
}

moe_status moe_expert_ffn_slots(const uint16_t* xp, const int32_t* group_offsets, const int32_t* group_slot, int G,
                                int n_slots, int A, const uint16_t* w1, const uint16_t* w3, const uint16_t* w2, int H,
                                int F, moe_act act, int small_group_threshold, uint16_t* y, void* workspace,
                                size_t ws_bytes, void* stream) {
  if (!group_slot) return fail(MOE_ERR_INVALID, "moe_expert_ffn_slots: null group_slot");
  return expert_ffn("moe_expert_ffn_slots", xp, nullptr, 1, 0, group_offsets, group_slot, G, nullptr, n_slots, A, w1,
                    w3, w2, H, F, act, small_group_threshold, y, workspace, ws_bytes, stream);
}

moe_status moe_replicate_weights(const int32_t* rep_base, int E, uint16_t* w_all, int rows, int cols,
                                 int32_t* group_slot, void* stream) {
  if (E < 1 || E > 256) return fail(MOE_ERR_INVALID, "moe_replicate_weights: need 1<=E<=256");
  if (!rep_base) return fail(MOE_ERR_INVALID, "moe_replicate_weights: null rep_base");
  if (w_all && (rows < 1 || cols < 1 || ((long long)rows * cols) % 8 != 0 || !aligned(w_all, 16)))
    return fail(MOE_ERR_INVALID, "moe_replicate_weights: rows*cols must be a positive multiple of 8, w_all 16-byte aligned");
  DeviceInfo* d = nullptr;
  moe_status ms = device_info(&d);
  if (ms != MOE_OK) return ms;
  return cuda_status(replica_copy::launch(rep_base, E, w_all, (long long)rows * cols, group_slot, d->num_sms,
                                          static_cast<cudaStream_t>(stream)),
                     "moe_replicate_weights launch");
}

int moe_ffn_launches(int A, int E, int H, int F, int act, int small_group_threshold, int gather) {
  // the sizes moe_expert_ffn accepts; anything it refuses launches nothing
  if (A <= 0 || E < 1 || E > ffn::MAX_G || H < 64 || H % 64 || F < 64 || F % 64) return 0;
  if ((act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU) || small_group_threshold < 0) return 0;
  bool use_pair = false, use_fused = false;
  ffn_choice(A, E, H, F, act, gather != 0, &use_pair, &use_fused);
  const bool small_path = small_group_threshold > 0 && g_opt_ffn_small_sms.load(std::memory_order_relaxed) != 0;
  return (use_fused ? 1 : 2) + (small_path ? 2 : 0);
}

// ------------------------------------------------------------------ options
moe_status moe_set_option(int option, int value) {
  if (option == MOE_OPT_FFN_KERNEL) {
    if (value < MOE_FFN_KERNEL_AUTO || value > MOE_FFN_KERNEL_FUSED)
      return fail(MOE_ERR_INVALID, "moe_set_option: unknown FFN kernel %d", value);
    g_opt_ffn_kernel.store(value);
    return MOE_OK;
  }
  if (option == MOE_OPT_PDL) {
    if (value != 0 && value != 1) return fail(MOE_ERR_INVALID, "moe_set_option: PDL value must be 0 or 1");
    g_moe_pdl.store(value);
    return MOE_OK;
  }
  if (option == MOE_OPT_FFN_TIMEOUT_SELFTEST) {
    if (value != 0 && value != 1) return fail(MOE_ERR_INVALID, "moe_set_option: self-test value must be 0 or 1");
    g_opt_ffn_selftest.store(value);
    return MOE_OK;
  }
  if (option == MOE_OPT_FFN_SMALL_SMS) {
    if (value < -1 || value > 4096) return fail(MOE_ERR_INVALID, "moe_set_option: small-path SMs must be -1..4096");
    g_opt_ffn_small_sms.store(value);
    return MOE_OK;
  }
  if (option == MOE_OPT_FRONT_ONE_LAUNCH) {
    if (value != 0 && value != 1) return fail(MOE_ERR_INVALID, "moe_set_option: one-launch front value must be 0 or 1");
    front::g_front_one_launch.store(value);
    return MOE_OK;
  }
  return fail(MOE_ERR_INVALID, "moe_set_option: unknown option %d", option);
}

moe_status moe_get_option(int option, int* value) {
  if (!value) return fail(MOE_ERR_INVALID, "moe_get_option: null value");
  if (option == MOE_OPT_FFN_KERNEL) {
    *value = g_opt_ffn_kernel.load();
    return MOE_OK;
  }
  if (option == MOE_OPT_PDL) {
    *value = g_moe_pdl.load();
    return MOE_OK;
  }
  if (option == MOE_OPT_FFN_TIMEOUT_SELFTEST) {
    *value = g_opt_ffn_selftest.load();
    return MOE_OK;
  }
  if (option == MOE_OPT_FFN_SMALL_SMS) {
    *value = g_opt_ffn_small_sms.load();
    return MOE_OK;
  }
  if (option == MOE_OPT_FRONT_ONE_LAUNCH) {
    *value = front::g_front_one_launch.load();
    return MOE_OK;
  }
  return fail(MOE_ERR_INVALID, "moe_get_option: unknown option %d", option);
}

int moe_layer_front_launches(int T, int E, int k, int has_prev) {
  if (T <= 0 || E < 1 || E > 256 || k < 1 || k > 8 || k > E) return 0;
  DeviceInfo* d = nullptr;
  if (device_info(&d) != MOE_OK) return 0;
  return front::launches(T, E, k, has_prev != 0, d->num_sms);
}

// ------------------------------------------------------------------ combine
moe_status moe_combine(const uint16_t* y, const int32_t* inv_perm, const float* w, int T, int k, int H, uint16_t* out,
                       void* stream) {
  if (T < 0 || k < 1 || k > 8 || H < 8 || H % 8)
    return fail(MOE_ERR_INVALID, "moe_combine: need T>=0, 1<=k<=8, H a positive multiple of 8");
  if ((long long)T * k >= (1LL << 31)) return fail(MOE_ERR_INVALID, "moe_combine: T*k too large");
  if (T == 0) return MOE_OK;
  if (!y || !inv_perm || !w || !out) return fail(MOE_ERR_INVALID, "moe_combine: null pointer");
  if (!aligned(y, 16) || !aligned(out, 16)) return fail(MOE_ERR_INVALID, "moe_combine: y/out must be 16-byte aligned");
  DeviceInfo* d = nullptr;
  moe_status ms = device_info(&d);
  if (ms != MOE_OK) return ms;
  return cuda_status(combine::launch(y, inv_perm, w, T, k, H, out, d->num_sms, static_cast<cudaStream_t>(stream)),
                     "moe_combine launch");
}

// ------------------------------------------------------------------ errors
moe_status moe_error_word(uint32_t* word_out) {
  if (!word_out) return fail(MOE_ERR_INVALID, "moe_error_word: null pointer");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e, "moe_error_word: sync");
  e = cudaMemcpyFromSymbol(word_out, g_moe_dev_error, sizeof(uint32_t));
  return cuda_status(e, "moe_error_word: read");
}

moe_status moe_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e, "moe_check: stream sync");
  uint32_t word = 0;
  e = cudaMemcpyFromSymbol(&word, g_moe_dev_error, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_status(e, "moe_check: read error word");
  if (word) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_moe_dev_error, &zero, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_status(e, "moe_check: clear error word");
    if (word & MOE_DEVERR_TIMEOUT) return fail(MOE_ERR_TIMEOUT, "a bounded device wait ran out (word 0x%x)", word);
    return fail(MOE_ERR_DEVICE, "a kernel met invalid device data (word 0x%x)", word);
  }
  e = cudaGetLastError();
  return cuda_status(e, "moe_check");
}

}  // extern "C"

// moe_dispatch_noalloc lives in its own file and is compiled into this
// translation unit.
#include "dispatch_noalloc.cu"

// The backward of the routed expert layer, likewise.
#include "ffn_backward.cu"
