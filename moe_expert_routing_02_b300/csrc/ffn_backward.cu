// moe_ffn_backward and moe_route_backward: the backward of the routed expert
// layer (expert FFN, combine, dispatch copy) and of the top-k gate.
//
// PopFetcher (ATC'25) review: the system trains MoE models; the backward of
// a replicated expert reduces the replicas' gradients into the primary
// expert (core method and design trade-offs).  Here every row of an expert,
// in whichever replica group it was served, adds into that expert's one
// gradient inside the weight-gradient GEMM.
//
// Steps (one stream, seven launches):
//   1 layout   padded row space of the expert units (bwd::layout_kernel)
//   2 gather   xp = x rows, dY = w * dout rows in that space, dw = <dout, y>
//   3 recompute GEMM1 with the backward epilogue:   (ffn::gemm_kernel<kBwd*>)
//              GeLU: a = gelu(z) and the factor gelu'(z);
//              SwiGLU: a = silu(g) u and the factors u silu'(g), silu(g)
//   4 dgrad    dA = dY W2^T, multiplied by the factors in the epilogue:
//              dz (GeLU) or [dg | du] (SwiGLU)  (ffn::gemm_kernel<kStoreKMMul>)
//   5 dgrad    dxp = dz W1^T  (SwiGLU: [dg du] [W1; W3]^T, K = 2F)
//   6 wgrad    dW2 = a^T dY, dW1 = xp^T dz (SwiGLU: dg), dW3 = xp^T du
//   7 scatter  dx[t] = sum_r dxp[row of (t, r)]
//
// This file is compiled as part of the library's single translation unit (it
// is included at the end of moe_api.cu).

#include "bwd.cuh"
#include "ffn_wgrad.cuh"

namespace {

// Workspace of moe_ffn_backward, for G = 2E groups and SwiGLU (the larger
// activation); offsets in bytes, each a multiple of 256.
struct BwdWs {
  long long P;  // rows of the padded row space (bound)
  size_t pgoff, pue, ustart, pbeg, pcnt, prow, xp, dy, act, dz, dxp, total;
};

BwdWs bwd_ws(long long A, int E, int H, int F) {
  BwdWs w{};
  const long long G = 2LL * E;
  w.P = A + 64 * G;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += (bytes + 255) & ~(size_t)255;
    return at;
  };
  w.pgoff = take((size_t)(G + 1) * 4);
  w.pue = take((size_t)G * 4);
  w.ustart = take((size_t)(G + 1) * 4);
  w.pbeg = take((size_t)E * 4);
  w.pcnt = take((size_t)E * 4);
  w.prow = take((size_t)(A > 0 ? A : 1) * 4);
  w.xp = take((size_t)w.P * H * 2);
  w.dy = take((size_t)w.P * H * 2);
  w.act = take((size_t)w.P * F * 2);
  w.dz = take((size_t)w.P * 2 * F * 2);
  w.dxp = take((size_t)w.P * H * 2);
  w.total = o;
  return w;
}

bool g_bwd_attr[kMaxDevices][6] = {};

moe_status bwd_attrs(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  const void* fns[6] = {(const void*)ffn::gemm_kernel<ffn::kStoreKM>,    (const void*)ffn::gemm_kernel<ffn::kBwdGelu>,
                        (const void*)ffn::gemm_kernel<ffn::kBwdSwiglu>,  (const void*)ffn_wg::wgrad_kernel,
                        (const void*)ffn::gemm_kernel<ffn::kStoreKMMul>, (const void*)ffn::gemm_kernel<ffn::kStoreKMMul2>};
  const int bytes[6] = {(int)ffn::kSmemBytes, (int)ffn::kSmemBytes, (int)ffn::kSmemBytes, (int)ffn_wg::kSmemBytes,
                        (int)ffn::kSmemBytes, (int)ffn::kSmemBytes};
  for (int i = 0; i < 6; ++i) {
    if (g_bwd_attr[dev][i]) continue;
    cudaError_t e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, bytes[i]);
    if (e != cudaSuccess) return cuda_at("moe_ffn_backward", e, "cudaFuncSetAttribute");
    g_bwd_attr[dev][i] = true;
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_ffn_backward_workspace_bytes(int T, int k, int E, int H, int F) {
  if (T < 0 || k < 1 || k > 8 || E < 1 || E > 256 || H < 64 || H % 64 || F < 64 || F % 64) return 0;
  return bwd_ws((long long)T * k, E, H, F).total;
}

moe_status moe_ffn_backward(const uint16_t* x, const uint16_t* dout, const float* w, const uint16_t* y,
                            const int32_t* perm, const int32_t* inv_perm, int T, int k, const int32_t* group_offsets,
                            const int32_t* group_expert, int E, const uint16_t* w1, const uint16_t* w3,
                            const uint16_t* w2, int H, int F, moe_act act, uint16_t* dx, float* dw, void* dw1,
                            void* dw3, void* dw2, int flags, void* workspace, size_t ws_bytes, void* stream) {
  const char* who = "moe_ffn_backward";
  if (T < 0 || k < 1 || k > 8 || E < 1 || E > 256 || k > E)
    return fail(MOE_ERR_INVALID, "%s: need T>=0, 1<=k<=min(E,8), 1<=E<=256", who);
  if (H < 64 || H % 64 || F < 64 || F % 64) return fail(MOE_ERR_INVALID, "%s: H and F must be positive multiples of 64", who);
  if (act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID, "%s: unknown activation", who);
  if (flags & ~(MOE_BWD_ACCUMULATE_WGRAD | MOE_BWD_WGRAD_BF16))
    return fail(MOE_ERR_INVALID, "%s: unknown flags 0x%x", who, flags);
  if ((flags & MOE_BWD_ACCUMULATE_WGRAD) && (flags & MOE_BWD_WGRAD_BF16))
    return fail(MOE_ERR_INVALID, "%s: bf16 weight gradients cannot be accumulated", who);
  const long long A = (long long)T * k;
  const BwdWs L = bwd_ws(A, E, H, F);
  if (L.P * 2 * F >= (1LL << 40) || L.P >= (1LL << 31) - 256 || (long long)E * H >= (1LL << 31) ||
      (long long)E * F >= (1LL << 31))
    return fail(MOE_ERR_INVALID, "%s: problem too large", who);
  if (!group_offsets || !w1 || !w2 || !dw1 || !dw2 || !workspace) return fail(MOE_ERR_INVALID, "%s: null pointer", who);
  if (act == MOE_ACT_SWIGLU && (!w3 || !dw3)) return fail(MOE_ERR_INVALID, "%s: SwiGLU needs w3 and dw3", who);
  if (T > 0 && (!x || !dout || !w || !perm || !inv_perm || !dx))
    return fail(MOE_ERR_INVALID, "%s: null pointer", who);
  if (y && !dw) return fail(MOE_ERR_INVALID, "%s: y given without dw", who);
  if (!aligned(w1, 16) || !aligned(w2, 16) || (w3 && !aligned(w3, 16)) || !aligned(dw1, 16) || !aligned(dw2, 16) ||
      (dw3 && !aligned(dw3, 16)) || (x && !aligned(x, 16)) || (dout && !aligned(dout, 16)) ||
      (y && !aligned(y, 16)) || (dx && !aligned(dx, 16)) || !aligned(workspace, 256))
    return fail(MOE_ERR_INVALID, "%s: matrices must be 16-byte aligned, the workspace 256-byte aligned", who);
  if (ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "%s: workspace needs %zu bytes", who, L.total);

  DeviceInfo* d = nullptr;
  moe_status ms = device_info(&d);
  if (ms != MOE_OK) return ms;
  if ((ms = get_encoder()) != MOE_OK) return ms;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
  if ((ms = bwd_attrs(dev)) != MOE_OK) return ms;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* pgoff = reinterpret_cast<int32_t*>(ws + L.pgoff);
  int32_t* pue = reinterpret_cast<int32_t*>(ws + L.pue);
  int32_t* ustart = reinterpret_cast<int32_t*>(ws + L.ustart);
  int32_t* pbeg = reinterpret_cast<int32_t*>(ws + L.pbeg);
  int32_t* pcnt = reinterpret_cast<int32_t*>(ws + L.pcnt);
  int32_t* prow = reinterpret_cast<int32_t*>(ws + L.prow);
  uint16_t* xp = reinterpret_cast<uint16_t*>(ws + L.xp);
  uint16_t* dy = reinterpret_cast<uint16_t*>(ws + L.dy);
  uint16_t* av = reinterpret_cast<uint16_t*>(ws + L.act);
  uint16_t* dz = reinterpret_cast<uint16_t*>(ws + L.dz);
  uint16_t* dxp = reinterpret_cast<uint16_t*>(ws + L.dxp);
  const bool swiglu = act == MOE_ACT_SWIGLU;
  const int G = group_expert ? 2 * E : E;
  const int KZ = swiglu ? 2 * F : F;  // columns of dz ([dg | du] for SwiGLU)
  const long long P = L.P;

  // ---- tensor maps
  CUtensorMap mDy, mW2k, mXp, mDz, mW1k, mW3k;
  if ((ms = encode_2d(&mDy, dy, H, P, 64, ffn::BM)) != MOE_OK) return ms;
  if ((ms = encode_2d(&mW2k, w2, H, (uint64_t)E * F, 64, ffn::BN)) != MOE_OK) return ms;
  if ((ms = encode_2d(&mXp, xp, H, P, 64, ffn::BM)) != MOE_OK) return ms;
  if ((ms = encode_2d(&mDz, dz, KZ, P, 64, ffn::BM)) != MOE_OK) return ms;
  if ((ms = encode_2d(&mW1k, w1, F, (uint64_t)E * H, 64, ffn::BN)) != MOE_OK) return ms;
  if ((ms = encode_2d(&mW3k, swiglu ? w3 : w1, F, (uint64_t)E * H, 64, ffn::BN)) != MOE_OK) return ms;
  ffn_wg::Maps wm;
  if ((ms = encode_2d(&wm.a[0], av, F, P, 64, 64)) != MOE_OK) return ms;
  if ((ms = encode_2d(&wm.b[0], dy, H, P, 64, 64)) != MOE_OK) return ms;
  if ((ms = encode_2d(&wm.a[1], xp, H, P, 64, 64)) != MOE_OK) return ms;
  if ((ms = encode_2d(&wm.b[1], dz, KZ, P, 64, 64)) != MOE_OK) return ms;
  wm.a[2] = wm.a[1];
  wm.b[2] = wm.b[1];

  // ---- 1, 2: layout and gather
  bwd::layout_kernel<<<1, bwd::kLayoutThreads, 0, st>>>(group_offsets, group_expert, G, E, (int)A, pgoff, pue, ustart,
                                                       pbeg, pcnt);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_at(who, e, "layout launch");
  {
    long long blocks = (P + 7) / 8;
    if (blocks > 16LL * d->num_sms) blocks = 16LL * d->num_sms;
    bwd::gather_kernel<<<(unsigned)blocks, 256, 0, st>>>(pgoff, ustart, G, perm, T, k, x, dout, w, y, H, xp, dy,
                                                          y ? dw : nullptr, prow);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_at(who, e, "gather launch");
  }

  // ---- 3..5: the data-gradient GEMMs over the padded units
  ffn::Params pb{};
  pb.group_offsets = pgoff;
  pb.group_expert = pue;
  pb.G = G;
  pb.E = E;
  pb.A_rows = P;
  pb.a_src_div = 1;
  const long long mt_bound = (P + ffn::BM - 1) / ffn::BM + G;
  auto grid_for = [&](const ffn::Params& p) {
    long long g = mt_bound * p.n_tiles;
    if (g > d->num_sms) g = d->num_sms;
    return (unsigned)(g < 1 ? 1 : g);
  };
  ffn::Params p4 = pb;  // GEMM1 recomputed: activation and derivative factors
  p4.K = H;
  p4.N_out = F;
  p4.n_tiles = swiglu ? (F + ffn::BN / 2 - 1) / (ffn::BN / 2) : (F + ffn::BN - 1) / ffn::BN;
  p4.out = av;
  p4.out2 = dz;
  // the weight tiles as one 3-D box per matrix and stage, as in the forward
  CUtensorMap mW1q, mW3q;
  if ((ms = encode_w3d(&mW1q, w1, F, (uint64_t)E * H, swiglu ? 2 : 4)) != MOE_OK) return ms;
  if ((ms = encode_w3d(&mW3q, swiglu ? w3 : w1, F, (uint64_t)E * H, swiglu ? 2 : 4)) != MOE_OK) return ms;
  p4.b3d = 1;
  if (swiglu)
    ffn::gemm_kernel<ffn::kBwdSwiglu><<<grid_for(p4), ffn::THREADS, ffn::kSmemBytes, st>>>(mXp, mW1q, mW3q, p4);
  else
    ffn::gemm_kernel<ffn::kBwdGelu><<<grid_for(p4), ffn::THREADS, ffn::kSmemBytes, st>>>(mXp, mW1q, mW3q, p4);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_at(who, e, "recompute launch");

  ffn::Params p3 = pb;  // dA = dY W2^T (K = H, N = F) times the factors, in place
  p3.K = H;
  p3.N_out = F;
  p3.n_tiles = (F + ffn::BN - 1) / ffn::BN;
  p3.k_split = H / ffn::BK;
  p3.out = dz;
  if (swiglu) {
    ffn::gemm_kernel<ffn::kStoreKMMul2><<<grid_for(p3), ffn::THREADS, ffn::kSmemBytes, st>>>(mDy, mW2k, mW2k, p3);
  } else {
    // the factor tiles come through TMA: 16-column x 32-row boxes of dz
    CUtensorMap mF;
    if ((ms = encode_2d(&mF, dz, F, P, 16, 32, false)) != MOE_OK) return ms;
    ffn::gemm_kernel<ffn::kStoreKMMul><<<grid_for(p3), ffn::THREADS, ffn::kSmemBytes, st>>>(mDy, mW2k, mF, p3);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_at(who, e, "dgrad (dA) launch");

  ffn::Params p5 = pb;  // dxp = dz W1^T (+ du W3^T): K = F or 2F, N = H
  p5.K = KZ;
  p5.N_out = H;
  p5.n_tiles = (H + ffn::BN - 1) / ffn::BN;
  p5.k_split = F / ffn::BK;
  p5.out = dxp;
  ffn::gemm_kernel<ffn::kStoreKM><<<grid_for(p5), ffn::THREADS, ffn::kSmemBytes, st>>>(mDz, mW1k, mW3k, p5);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_at(who, e, "dgrad (dx) launch");

  // ---- 6: weight gradients, all jobs in one launch
  ffn_wg::WParams wp{};
  wp.pbeg = pbeg;
  wp.pcnt = pcnt;
  wp.E = E;
  wp.rows = P;
  wp.jobs = swiglu ? 3 : 2;
  wp.accumulate = (flags & MOE_BWD_ACCUMULATE_WGRAD) ? 1 : 0;
  wp.out_bf16 = (flags & MOE_BWD_WGRAD_BF16) ? 1 : 0;
  auto job = [&](ffn_wg::Job& j, void* out, int M, int N, int b_col0) {
    j.out = out;
    j.M_out = M;
    j.N_out = N;
    j.m_tiles = (M + ffn::BM - 1) / ffn::BM;
    j.n_tiles = (N + ffn::BN - 1) / ffn::BN;
    j.a_col0 = 0;
    j.b_col0 = b_col0;
  };
  job(wp.job[0], dw2, F, H, 0);
  job(wp.job[1], dw1, H, F, 0);
  if (swiglu) job(wp.job[2], dw3, H, F, F);
  wp.tiles_per_expert = 0;
  for (int j = 0; j < wp.jobs; ++j) wp.tiles_per_expert += wp.job[j].m_tiles * wp.job[j].n_tiles;
  {
    long long g = (long long)E * wp.tiles_per_expert;
    if (g > d->num_sms) g = d->num_sms;
    ffn_wg::wgrad_kernel<<<(unsigned)g, ffn::THREADS, ffn_wg::kSmemBytes, st>>>(wm, wp);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_at(who, e, "wgrad launch");
  }

  // ---- 7: token gradient
  if (T > 0) {
    long long blocks = ((long long)T + 7) / 8;
    if (blocks > 16LL * d->num_sms) blocks = 16LL * d->num_sms;
    bwd::scatter_kernel<<<(unsigned)blocks, 256, 0, st>>>(dxp, prow, inv_perm, T, k, H, P, dx);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_at(who, e, "scatter launch");
  }
  return MOE_OK;
}

moe_status moe_route_backward(const float* logits, const int32_t* idx, const float* dw, int T, int E, int k,
                              int renorm, float* dlogits, void* stream) {
  if (T < 0 || E < 1 || E > 256 || k < 1 || k > 8 || k > E)
    return fail(MOE_ERR_INVALID, "moe_route_backward: need T>=0, 1<=k<=min(E,8), E<=256");
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !dw || !dlogits) return fail(MOE_ERR_INVALID, "moe_route_backward: null pointer");
  DeviceInfo* d = nullptr;
  moe_status ms = device_info(&d);
  if (ms != MOE_OK) return ms;
  long long blocks = ((long long)T + 255) / 256;
  if (blocks > 16LL * d->num_sms) blocks = 16LL * d->num_sms;
  bwd::route_bwd_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(logits, idx, dw, T, E, k,
                                                                                         renorm ? 1 : 0, dlogits);
  return cuda_status(cudaGetLastError(), "moe_route_backward launch");
}

}  // extern "C"
