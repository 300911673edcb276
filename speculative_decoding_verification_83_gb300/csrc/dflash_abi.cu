// dflash_abi.cu -- the extern "C" entry points declared in include/dflash_verify.h:
// argument checks, workspace layout, launch configuration and the host-buffer
// path. No device memory is allocated here; every buffer belongs to the caller.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/dflash_verify.h"
#include "dflash_internal.h"

using namespace dflash;

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

// An NVTX range around an entry point's host work and launches, so that a
// timeline profiler shows each call by name (a no-op without a profiler).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DFLASH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// SMs the calling thread's current context may use: all of the device's
// for a primary context, the partition's for a green context (from the
// driver's resource query, reached through the runtime so the library does
// not link the driver). Cached per context.
typedef int (*CtxGetCurrentFn)(CUcontext*);
typedef int (*CtxGetDevResourceFn)(CUcontext, CUdevResource*, CUdevResourceType);

int available_sms(int dev) {
  static std::mutex mu;
  static bool looked_up = false;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetDevResourceFn get_resource = nullptr;
  static CUcontext ctx_cache[kMaxDevices * 4] = {};
  static int sms_cache[kMaxDevices * 4] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!looked_up) {
    looked_up = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12040, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetDevResource", &f, 12040, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_resource = reinterpret_cast<CtxGetDevResourceFn>(f);
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  CUcontext ctx = nullptr;
  if (!get_current || !get_resource || get_current(&ctx) != 0 || !ctx) return n;
  for (int i = 0; i < kMaxDevices * 4 && ctx_cache[i]; ++i)
    if (ctx_cache[i] == ctx) return sms_cache[i];
  CUdevResource res;
  memset(&res, 0, sizeof res);
  if (get_resource(ctx, &res, CU_DEV_RESOURCE_TYPE_SM) == 0 && res.sm.smCount > 0 &&
      (int)res.sm.smCount < n)
    n = (int)res.sm.smCount;
  for (int i = 0; i < kMaxDevices * 4; ++i)
    if (!ctx_cache[i]) {
      ctx_cache[i] = ctx;
      sms_cache[i] = n;
      break;
    }
  return n;
}

int esize_of(int dtype) { return dtype == DFLASH_BF16 ? 2 : (dtype == DFLASH_F32 ? 4 : 0); }

// Filter mode of a call: 1 = top-k (1..32) with any top_p, 2 = full
// vocabulary (top-k off, top_p >= 1), 3 = top-p over the full vocabulary
// (top-k off, top_p < 1), 0 = unsupported, -1 = invalid.
constexpr int kModeTopK = 1, kModeFullVocab = 2, kModeFullVocabTopP = 3;
// The top-p cut over the full vocabulary sums fixed-point weights in 64 bits
// with 62 - ceil(log2 V) fractional bits: the sums' error, as a fraction of
// the row's mass, is below V^2 2^-62, which stays under 2^-18 up to 2^22 tokens.
constexpr int kFvtpMaxV = 1 << 22;
int filter_mode(int V, int top_k, float top_p) {
  if (!(top_p > 0.0f) || std::isnan(top_p)) return -1;
  const bool k_on = top_k > 0 && top_k < V;
  if (k_on && top_k <= DFLASH_MAX_TOP_K) return kModeTopK;
  if (!k_on && top_p >= 1.0f) return kModeFullVocab;
  if (!k_on && V <= kFvtpMaxV) return kModeFullVocabTopP;
  return 0;
}
bool whole_vocab(int mode) { return mode == kModeFullVocab || mode == kModeFullVocabTopP; }

// 2^(j/64), j < 64, split into fp32 pairs (hi = nearest float, lo = the rest)
// for the full-vocabulary draw's exp; computed once in double precision.
struct Exp2Table {
  float hi[kExpTable], lo[kExpTable];
  Exp2Table() {
    for (int j = 0; j < kExpTable; ++j) {
      const double v = std::exp2((double)j / kExpTable);
      hi[j] = (float)v;
      lo[j] = (float)(v - (double)hi[j]);
    }
  }
};
const Exp2Table& exp2_table() {
  static const Exp2Table t;
  return t;
}

int check_shape(int B, int gamma, int V, int dtype) {
  if (B < 1 || B > kMaxB) return fail(DFLASH_ERR_INVALID_ARG, "B=%d outside [1, %d]", B, kMaxB);
  if (gamma < 1 || gamma > kMaxGamma)
    return fail(DFLASH_ERR_INVALID_ARG, "gamma=%d outside [1, %d]", gamma, kMaxGamma);
  if (V < 1) return fail(DFLASH_ERR_INVALID_ARG, "V=%d must be >= 1", V);
  if (!esize_of(dtype)) return fail(DFLASH_ERR_INVALID_ARG, "dtype=%d is neither bf16 nor fp32", dtype);
  return DFLASH_OK;
}

int check_aligned(const void* p, int esize, const char* name) {
  if (((uintptr_t)p) % (uintptr_t)esize)
    return fail(DFLASH_ERR_INVALID_ARG, "%s is not aligned to its element size", name);
  return DFLASH_OK;
}

size_t verify_workspace(int B, int gamma, int V, int dtype, int mode = kModeTopK) {
  const Geometry g = make_geometry(V, esize_of(dtype));
  return make_layout(B * (2 * gamma + 1), B, g, whole_vocab(mode), mode == kModeFullVocabTopP).total;
}

void bind_workspace(Params& p, void* ws, int n_slots, int n_requests, int mode = kModeTopK) {
  const bool fullvocab = whole_vocab(mode);
  const WorkspaceLayout L = make_layout(n_slots, n_requests, p.geo, fullvocab, mode == kModeFullVocabTopP);
  unsigned char* base = static_cast<unsigned char*>(ws);
  p.row_cnt = reinterpret_cast<uint32_t*>(base + L.row_cnt);
  p.abort_flag = reinterpret_cast<uint32_t*>(base + L.abort_flag);
  p.job_cnt = p.abort_flag + 1;
  p.row_best = reinterpret_cast<unsigned long long*>(base + L.row_best);
  p.tile_keys = reinterpret_cast<uint32_t*>(base + L.tile_keys);
  p.res_list = reinterpret_cast<unsigned long long*>(base + L.res_list);
  p.fv_draw = fullvocab ? reinterpret_cast<FvDraw*>(base + L.fv_draw) : nullptr;
  p.fullvocab = fullvocab ? 1 : 0;
  p.fvtp = mode == kModeFullVocabTopP ? 1 : 0;
  p.fvtp_rows = p.fvtp ? reinterpret_cast<float4*>(base + L.tp_rows) : nullptr;
  p.n_slots = n_slots;
}

int ceil_log2(long long v) {
  int c = 0;
  while ((1ll << c) < v) ++c;
  return c;
}

// top-p over the full vocabulary: the rows' cuts and the accept tests, between
// the stream and the draw
int run_fvtp(const Params& p, void* ws, void* stream, bool sampler) {
  const WorkspaceLayout L = make_layout(p.n_slots, p.B, p.geo, true, true);
  unsigned char* base = static_cast<unsigned char*>(ws);
  FvtpParams t;
  memset(&t, 0, sizeof t);
  t.target = p.target;
  t.draft = p.draft;
  t.draft_tokens = p.draft_tokens;
  t.temperature = p.temperature;
  t.B = p.B;
  t.gamma = p.gamma;
  t.V = p.geo.V;
  t.dtype = p.dtype;
  t.det = p.det;
  t.per_s = p.det ? p.gamma + 1 : 2 * p.gamma + 1;
  t.n_slices = fv_slices(p.geo.V);
  t.frac_bits = 62 - ceil_log2(p.geo.V);  // the row's mass, at most V, fits 63 bits
  t.top_p = p.top_p;
  t.seed = p.seed;
  t.sampler = sampler ? 1 : 0;
  t.row_base = p.row_base;
  t.out_tokens = p.out_tokens;
  t.out_len = p.out_len;
  t.status = p.status;
  t.audit_pq = p.audit_pq;
  t.rows = reinterpret_cast<float4*>(base + L.tp_rows);
  t.cut = reinterpret_cast<FvtpCut*>(base + L.tp_cut);
  t.hist_m = reinterpret_cast<unsigned long long*>(base + L.tp_hist_m);
  t.kcount = reinterpret_cast<uint32_t*>(base + L.tp_kcount);
  t.draw = reinterpret_cast<FvDraw*>(base + L.fv_draw);
  t.draw_cut = reinterpret_cast<FvtpDrawCut*>(base + L.tp_draw);
  t.abort_flag = p.abort_flag;
  t.exp2 = p.exp2;
  const int e = launch_fvtp_cut(t, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "launching the top-p cut over the full vocabulary");
  return DFLASH_OK;
}

// the full-vocabulary draw's second pass over the rows the accept test left
int run_fullvocab_draw(const Params& p, void* ws, void* stream, bool sampler = false) {
  const WorkspaceLayout L = make_layout(p.n_slots, p.B, p.geo, true, p.fvtp != 0);
  unsigned char* base = static_cast<unsigned char*>(ws);
  FvParams f;
  memset(&f, 0, sizeof f);
  f.target = p.target;
  f.draft = p.draft;
  f.temperature = p.temperature;
  f.B = p.B;
  f.gamma = p.gamma;
  f.V = p.geo.V;
  f.dtype = p.dtype;
  f.n_slices = fv_slices(p.geo.V);
  f.seed = p.seed;
  f.out_tokens = p.out_tokens;
  f.draw = reinterpret_cast<const FvDraw*>(base + L.fv_draw);
  f.part = reinterpret_cast<float4*>(base + L.fv_part);
  f.pos = reinterpret_cast<float4*>(base + L.fv_pos);
  f.last = reinterpret_cast<int2*>(base + L.fv_last);
  f.abort_flag = p.abort_flag;
  f.sampler = sampler ? 1 : 0;
  f.row_base = p.row_base;
  f.cut = p.fvtp ? reinterpret_cast<FvtpDrawCut*>(base + L.tp_draw) : nullptr;
  const Exp2Table& t = exp2_table();
  memcpy(f.exp_hi, t.hi, sizeof t.hi);
  memcpy(f.exp_lo, t.lo, sizeof t.lo);
  const int e = launch_fullvocab_draw(f, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "launching the full-vocabulary draw");
  return DFLASH_OK;
}

int run(Params& p, int total_slots, void* stream) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "no CUDA device");
  if (dev < 0 || dev >= kMaxDevices) return fail(DFLASH_ERR_CUDA, "device %d beyond the supported %d", dev, kMaxDevices);
  int per_sm = 0;
  const int e_occ = sweep_occupancy(p.dtype, dev, &per_sm);
  if (e_occ != 0) return cuda_fail((cudaError_t)e_occ, "sizing the verification kernel");
  const int sms = available_sms(dev);
  const long long pieces = (long long)total_slots * p.geo.ppr;
  const long long grid = persistent_grid(pieces, sms, per_sm < kCtasPerSm ? per_sm : kCtasPerSm);
  if (grid < 1)
    return fail(DFLASH_ERR_CUDA, "the verification kernel does not fit on this device's SMs (%d SMs, %d CTAs each)",
                sms, per_sm);
  const int e = launch_sweep(p, (int)grid, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "launching the verification kernel");
  return DFLASH_OK;
}

// the stream, then (top-p over the full vocabulary) the cut and accept
// kernels, then (either full-vocabulary mode) the draw
int run_step(Params& p, int total_slots, void* ws, void* stream, bool sampler = false) {
  int rc = run(p, total_slots, stream);
  if (rc || !p.fullvocab) return rc;
  if (p.fvtp && (rc = run_fvtp(p, ws, stream, sampler))) return rc;
  return run_fullvocab_draw(p, ws, stream, sampler);
}

Params base_params(int dtype, int V) {
  Params p;
  memset(&p, 0, sizeof p);
  p.dtype = dtype == DFLASH_BF16 ? 0 : 1;
  p.geo = make_geometry(V, esize_of(dtype));
  const Exp2Table& e = exp2_table();
  memcpy(p.exp2.hi, e.hi, sizeof e.hi);
  memcpy(p.exp2.lo, e.lo, sizeof e.lo);
  return p;
}

}  // namespace

void dflash::set_last_error(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

extern "C" {

int dflash_abi_version(void) { return DFLASH_ABI_VERSION; }

const char* dflash_last_error(void) { return g_last_error; }

size_t dflash_workspace_bytes(int B, int gamma, int V, int dtype, int top_k, float top_p) {
  if (B < 1 || B > kMaxB || gamma < 1 || gamma > kMaxGamma || V < 1 || !esize_of(dtype)) return 0;
  const int mode = filter_mode(V, top_k, top_p);
  if (mode <= 0 && !(top_k == 1 && top_p >= 1.0f)) return 0;
  return verify_workspace(B, gamma, V, dtype, mode > 0 ? mode : kModeTopK);
}

size_t dflash_rows_workspace_bytes(int R, int V, int dtype, int top_k, float top_p) {
  if (R < 1 || V < 1 || !esize_of(dtype)) return 0;
  const int mode = filter_mode(V, top_k, top_p);
  if (whole_vocab(mode)) {  // the sampler over the full vocabulary: rows of kMaxB at a time
    const int chunk = R < kMaxB ? R : kMaxB;
    return verify_workspace(chunk, 0, V, dtype, mode);
  }
  if (mode != kModeTopK) return 0;
  const int chunk = R < kMaxCounterSlots ? R : kMaxCounterSlots;
  return make_layout(chunk, 1, make_geometry(V, esize_of(dtype))).total;
}

int dflash_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace && bytes) return fail(DFLASH_ERR_INVALID_ARG, "null workspace");
  if (!bytes) return DFLASH_OK;
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace");
  return DFLASH_OK;
}

int dflash_workspace_cancel(void* workspace, size_t bytes, void* stream) {
  // the abort flag sits in the workspace's fixed header, at the same offset
  // for every shape
  const size_t off = make_layout(1, 1, make_geometry(1, 4)).abort_flag;
  if (!workspace || bytes < off + sizeof(uint32_t))
    return fail(DFLASH_ERR_INVALID_ARG, "workspace of %zu bytes has no abort flag", bytes);
  cudaError_t e = cudaMemsetAsync(static_cast<unsigned char*>(workspace) + off, 1, sizeof(uint32_t),
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "setting the abort flag");
  return DFLASH_OK;
}

}  // extern "C"

namespace {
// dflash_verify, and with audit_pq the accept tests' p(d), q(d) written out
int verify_impl(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens, int B,
                int gamma, int V, int dtype, const float* temperature, int top_k, float top_p, uint64_t seed,
                int32_t* out_tokens, int32_t* out_accept_len, void* workspace, size_t workspace_bytes,
                uint32_t* status, float* audit_pq, void* stream) {
  int rc = check_shape(B, gamma, V, dtype);
  if (rc) return rc;
  if (!target_logits || !draft_logits || !draft_tokens || !temperature || !out_tokens || !out_accept_len ||
      !workspace)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  const int mode = filter_mode(V, top_k, top_p);
  if (mode < 0) return fail(DFLASH_ERR_INVALID_ARG, "top_p=%g must be in (0, 1]", (double)top_p);
  if (mode == 0)
    return fail(DFLASH_ERR_UNSUPPORTED,
                "top_k=%d with top_p=%g is not supported (need 1 <= top_k <= %d and top_k < V, or top-k off; "
                "top-k off with top_p < 1 needs V <= %d)",
                top_k, (double)top_p, DFLASH_MAX_TOP_K, kFvtpMaxV);
  const int es = esize_of(dtype);
  if ((rc = check_aligned(target_logits, es, "target_logits")) ||
      (rc = check_aligned(draft_logits, es, "draft_logits")))
    return rc;
  const size_t need = verify_workspace(B, gamma, V, dtype, mode);
  if (workspace_bytes < need)
    return fail(DFLASH_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, need);
  Params p = base_params(dtype, V);
  p.target = static_cast<const unsigned char*>(target_logits);
  p.draft = static_cast<const unsigned char*>(draft_logits);
  p.draft_tokens = draft_tokens;
  p.temperature = temperature;
  p.B = B;
  p.gamma = gamma;
  p.top_k = top_k;
  p.top_p = top_p >= 1.0f ? 1.0f : top_p;
  p.seed = seed;
  p.task = kTaskVerify;
  p.out_tokens = out_tokens;
  p.out_len = out_accept_len;
  p.audit_pq = audit_pq;
  p.status = status;
  bind_workspace(p, workspace, B * (2 * gamma + 1), B, mode);
  // the slot count depends on the device-side temperatures; launch for the maximum
  return run_step(p, B * (2 * gamma + 1), workspace, stream);
}

// ---- the LM head on the tensor cores ---------------------------------------------------
int check_lmhead(const void* h, const void* w, int M, int V, int K, const void* logits) {
  if (!h || !w || !logits) return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  if (M < 1 || M > kLmMaxRows) return fail(DFLASH_ERR_INVALID_ARG, "M=%d outside [1, %d]", M, kLmMaxRows);
  if (V < 8 || V % 8) return fail(DFLASH_ERR_INVALID_ARG, "V=%d must be a positive multiple of 8", V);
  if (K < 64 || K % 64) return fail(DFLASH_ERR_INVALID_ARG, "K=%d must be a positive multiple of 64", K);
  if (((uintptr_t)h | (uintptr_t)w | (uintptr_t)logits) % 16u)
    return fail(DFLASH_ERR_INVALID_ARG, "h, W and logits must be 16-byte aligned");
  return DFLASH_OK;
}
int lmhead_grid(int V, int* grid) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "no CUDA device");
  const int tiles = (V + 127) / 128, sms = available_sms(dev);
  *grid = tiles < sms ? tiles : sms;
  return DFLASH_OK;
}
}  // namespace

extern "C" {

int dflash_lmhead_logits(const void* h, const void* w, int M, int V, int K, void* logits, uint32_t* status,
                         void* stream) {
  NvtxRange nvtx_range("dflash_lmhead_logits");
  int rc = check_lmhead(h, w, M, V, K, logits);
  int grid = 0;
  if (rc || (rc = lmhead_grid(V, &grid))) return rc;
  LmParams lp;
  memset(&lp, 0, sizeof lp);
  lp.M = M;
  lp.Mt = M;
  lp.V = V;
  lp.K = K;
  lp.logits = static_cast<uint16_t*>(logits);
  lp.status = status;
  const int e = launch_lmhead(lp, h, w, false, grid, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "launching the LM head");
  return DFLASH_OK;
}

int dflash_lmhead_verify(const void* h, const void* w, int B, int gamma, int V, int K, const int32_t* draft_tokens,
                         const float* temperature, int top_k, float top_p, uint64_t seed, void* logits,
                         int32_t* out_tokens, int32_t* out_accept_len, void* workspace, size_t workspace_bytes,
                         uint32_t* status, void* stream) {
  NvtxRange nvtx_range("dflash_lmhead_verify");
  int rc = check_shape(B, gamma, V, DFLASH_BF16);
  if (rc) return rc;
  const long long M = (long long)B * (2 * gamma + 1);
  if (M > kLmMaxRows)
    return fail(DFLASH_ERR_INVALID_ARG, "B=%d gamma=%d gives %lld rows, more than the LM head's %d", B, gamma, M,
                kLmMaxRows);
  if ((rc = check_lmhead(h, w, (int)M, V, K, logits))) return rc;
  if (!draft_tokens || !temperature || !out_tokens || !out_accept_len || !workspace)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  const int mode = filter_mode(V, top_k, top_p);
  if (mode < 0) return fail(DFLASH_ERR_INVALID_ARG, "top_p=%g must be in (0, 1]", (double)top_p);
  if (mode != kModeTopK)
    return fail(DFLASH_ERR_UNSUPPORTED,
                "top_k=%d with top_p=%g is not supported in the LM head's epilogue (need 1 <= top_k <= %d and "
                "top_k < V)",
                top_k, (double)top_p, DFLASH_MAX_TOP_K);
  const size_t need = verify_workspace(B, gamma, V, DFLASH_BF16, mode);
  if (workspace_bytes < need)
    return fail(DFLASH_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, need);
  int grid = 0;
  if ((rc = lmhead_grid(V, &grid))) return rc;
  const int Mt = B * (gamma + 1);
  Params p = base_params(DFLASH_BF16, V);
  p.target = static_cast<const unsigned char*>(logits);
  p.draft = static_cast<const unsigned char*>(logits) + (size_t)Mt * V * 2;
  p.draft_tokens = draft_tokens;
  p.temperature = temperature;
  p.B = B;
  p.gamma = gamma;
  p.top_k = top_k;
  p.top_p = top_p >= 1.0f ? 1.0f : top_p;
  p.seed = seed;
  p.task = kTaskVerify;
  p.out_tokens = out_tokens;
  p.out_len = out_accept_len;
  p.status = status;
  p.keys_ready = 1;
  bind_workspace(p, workspace, B * (2 * gamma + 1), B, mode);
  LmParams lp;
  memset(&lp, 0, sizeof lp);
  lp.M = (int)M;
  lp.Mt = Mt;
  lp.V = V;
  lp.K = K;
  lp.logits = static_cast<uint16_t*>(logits);
  lp.B = B;
  lp.gamma = gamma;
  lp.tiles = p.geo.tiles;
  lp.temperature = temperature;
  lp.tile_keys = p.tile_keys;
  lp.row_best = p.row_best;
  lp.status = status;
  const int e = launch_lmhead(lp, h, w, true, grid, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "launching the LM head");
  return run(p, B * (2 * gamma + 1), stream);
}

int dflash_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens, int B,
                  int gamma, int V, int dtype, const float* temperature, int top_k, float top_p,
                  uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len, void* workspace,
                  size_t workspace_bytes, uint32_t* status, void* stream) {
  NvtxRange nvtx_range("dflash_verify");
  return verify_impl(target_logits, draft_logits, draft_tokens, B, gamma, V, dtype, temperature, top_k, top_p,
                     seed, out_tokens, out_accept_len, workspace, workspace_bytes, status, nullptr, stream);
}

int dflash_verify_audit(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                        int B, int gamma, int V, int dtype, const float* temperature, int top_k, float top_p,
                        uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len, float* audit_pq,
                        void* workspace, size_t workspace_bytes, uint32_t* status, void* stream) {
  NvtxRange nvtx_range("dflash_verify_audit");
  if (!audit_pq) return fail(DFLASH_ERR_INVALID_ARG, "null audit_pq");
  if (((uintptr_t)audit_pq) % 4u) return fail(DFLASH_ERR_INVALID_ARG, "audit_pq is not 4-byte aligned");
  return verify_impl(target_logits, draft_logits, draft_tokens, B, gamma, V, dtype, temperature, top_k, top_p,
                     seed, out_tokens, out_accept_len, workspace, workspace_bytes, status, audit_pq, stream);
}

int dflash_verify_det(const void* target_logits, const int32_t* draft_tokens, int B, int gamma, int V,
                      int dtype, const float* temperature, int top_k, float top_p, uint64_t seed,
                      int32_t* out_tokens, int32_t* out_accept_len, void* workspace, size_t workspace_bytes,
                      uint32_t* status, void* stream) {
  NvtxRange nvtx_range("dflash_verify_det");
  int rc = check_shape(B, gamma, V, dtype);
  if (rc) return rc;
  if (!target_logits || !draft_tokens || !temperature || !out_tokens || !out_accept_len || !workspace)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  const int mode = filter_mode(V, top_k, top_p);
  if (mode < 0) return fail(DFLASH_ERR_INVALID_ARG, "top_p=%g must be in (0, 1]", (double)top_p);
  if (mode == 0)
    return fail(DFLASH_ERR_UNSUPPORTED,
                "top_k=%d with top_p=%g is not supported for deterministic drafts (need 1 <= top_k <= %d "
                "and top_k < V, or top-k off)",
                top_k, (double)top_p, DFLASH_MAX_TOP_K);
  if ((rc = check_aligned(target_logits, esize_of(dtype), "target_logits"))) return rc;
  const size_t need = verify_workspace(B, gamma, V, dtype, mode);
  if (workspace_bytes < need)
    return fail(DFLASH_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, need);
  Params p = base_params(dtype, V);
  p.target = static_cast<const unsigned char*>(target_logits);
  p.draft_tokens = draft_tokens;
  p.temperature = temperature;
  p.B = B;
  p.gamma = gamma;
  p.top_k = top_k;
  p.top_p = top_p >= 1.0f ? 1.0f : top_p;
  p.seed = seed;
  p.task = kTaskVerify;
  p.det = 1;
  p.out_tokens = out_tokens;
  p.out_len = out_accept_len;
  p.status = status;
  bind_workspace(p, workspace, B * (gamma + 1), B, mode);
  return run_step(p, B * (gamma + 1), workspace, stream);  // reads target rows only: no residual mode here
}

int dflash_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int gamma, int V,
                         int dtype, int32_t* out_tokens, int32_t* out_accept_len, void* workspace,
                         size_t workspace_bytes, uint32_t* status, void* stream) {
  NvtxRange nvtx_range("dflash_verify_greedy");
  int rc = check_shape(B, gamma, V, dtype);
  if (rc) return rc;
  if (!target_logits || !draft_tokens || !out_tokens || !out_accept_len || !workspace)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  if ((rc = check_aligned(target_logits, esize_of(dtype), "target_logits"))) return rc;
  if (workspace_bytes < verify_workspace(B, gamma, V, dtype))
    return fail(DFLASH_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, verify_workspace(B, gamma, V, dtype));
  Params p = base_params(dtype, V);
  p.target = static_cast<const unsigned char*>(target_logits);
  p.draft_tokens = draft_tokens;
  p.B = B;
  p.gamma = gamma;
  p.top_k = 1;
  p.top_p = 1.0f;
  p.task = kTaskVerifyGreedy;
  p.out_tokens = out_tokens;
  p.out_len = out_accept_len;
  p.status = status;
  bind_workspace(p, workspace, B * (2 * gamma + 1), B);
  return run(p, B * (gamma + 1), stream);
}

size_t dflash_host_staging_bytes(int B, int gamma, int V, int dtype) {
  const int es = esize_of(dtype);
  if (B < 1 || gamma < 1 || V < 1 || !es) return 0;
  const size_t row = (size_t)V * es;
  size_t off = 0;
  off = align_up(off + row * (size_t)B * (gamma + 1), 256);  // target
  off = align_up(off + row * (size_t)B * gamma, 256);        // draft
  off = align_up(off + sizeof(int32_t) * (size_t)B * gamma, 256);
  off = align_up(off + sizeof(float) * (size_t)B, 256);
  off = align_up(off + sizeof(int32_t) * (size_t)B * (gamma + 1), 256);
  off = align_up(off + sizeof(int32_t) * (size_t)B, 256);
  off = align_up(off + sizeof(uint32_t), 256);
  return off;
}

int dflash_verify_host(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens, int B,
                       int gamma, int V, int dtype, const float* temperature, int top_k, float top_p,
                       uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len, uint32_t* out_status,
                       void* staging, size_t staging_bytes, void* workspace, size_t workspace_bytes,
                       void* stream) {
  NvtxRange nvtx_range("dflash_verify_host");
  int rc = check_shape(B, gamma, V, dtype);
  if (rc) return rc;
  if (!target_logits || !draft_logits || !draft_tokens || !temperature || !out_tokens || !out_accept_len ||
      !staging || !workspace)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  if (staging_bytes < dflash_host_staging_bytes(B, gamma, V, dtype))
    return fail(DFLASH_ERR_INVALID_ARG, "staging buffer too small");
  const int es = esize_of(dtype);
  const size_t row = (size_t)V * es;
  unsigned char* s = static_cast<unsigned char*>(staging);
  size_t off = 0;
  unsigned char* d_target = s + off;
  off = align_up(off + row * (size_t)B * (gamma + 1), 256);
  unsigned char* d_draft = s + off;
  off = align_up(off + row * (size_t)B * gamma, 256);
  int32_t* d_tokens_in = reinterpret_cast<int32_t*>(s + off);
  off = align_up(off + sizeof(int32_t) * (size_t)B * gamma, 256);
  float* d_temp = reinterpret_cast<float*>(s + off);
  off = align_up(off + sizeof(float) * (size_t)B, 256);
  int32_t* d_out = reinterpret_cast<int32_t*>(s + off);
  off = align_up(off + sizeof(int32_t) * (size_t)B * (gamma + 1), 256);
  int32_t* d_len = reinterpret_cast<int32_t*>(s + off);
  off = align_up(off + sizeof(int32_t) * (size_t)B, 256);
  uint32_t* d_status = reinterpret_cast<uint32_t*>(s + off);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
#define DFLASH_TRY(call, what)                       \
  do {                                               \
    e = (call);                                      \
    if (e != cudaSuccess) return cuda_fail(e, what); \
  } while (0)
  DFLASH_TRY(cudaMemcpyAsync(d_target, target_logits, row * (size_t)B * (gamma + 1), cudaMemcpyHostToDevice, st),
             "copying target logits");
  // draft rows: only requests that sample read them; copy runs of such requests
  for (int b = 0; b < B;) {
    const float t = temperature[b];
    if (!(t > 0.0f && std::isfinite(t))) {
      ++b;
      continue;
    }
    int e_b = b + 1;
    while (e_b < B && temperature[e_b] > 0.0f && std::isfinite(temperature[e_b])) ++e_b;
    const size_t off_b = row * (size_t)b * gamma, bytes = row * (size_t)(e_b - b) * gamma;
    DFLASH_TRY(cudaMemcpyAsync(d_draft + off_b, static_cast<const unsigned char*>(draft_logits) + off_b, bytes,
                               cudaMemcpyHostToDevice, st),
               "copying draft logits");
    b = e_b;
  }
  DFLASH_TRY(cudaMemcpyAsync(d_tokens_in, draft_tokens, sizeof(int32_t) * (size_t)B * gamma,
                             cudaMemcpyHostToDevice, st),
             "copying draft tokens");
  DFLASH_TRY(cudaMemcpyAsync(d_temp, temperature, sizeof(float) * (size_t)B, cudaMemcpyHostToDevice, st),
             "copying temperatures");
  DFLASH_TRY(cudaMemsetAsync(d_status, 0, sizeof(uint32_t), st), "clearing the status word");
  rc = dflash_verify(d_target, d_draft, d_tokens_in, B, gamma, V, dtype, d_temp, top_k, top_p, seed, d_out, d_len,
                     workspace, workspace_bytes, d_status, stream);
  if (rc) return rc;
  DFLASH_TRY(cudaMemcpyAsync(out_tokens, d_out, sizeof(int32_t) * (size_t)B * (gamma + 1),
                             cudaMemcpyDeviceToHost, st),
             "copying tokens back");
  DFLASH_TRY(cudaMemcpyAsync(out_accept_len, d_len, sizeof(int32_t) * (size_t)B, cudaMemcpyDeviceToHost, st),
             "copying accept lengths back");
  if (out_status)
    DFLASH_TRY(cudaMemcpyAsync(out_status, d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost, st),
               "copying the status back");
  DFLASH_TRY(cudaStreamSynchronize(st), "waiting for the stream");
#undef DFLASH_TRY
  return DFLASH_OK;
}

// The sampler over the full vocabulary (top-k off, top_p = 1) is the full-
// vocabulary verification with no draft positions: each row is a request
// whose only row is its bonus row, drawn from the whole softmax (T = 0: the
// argmax), with the sampler's uniforms. Rows go kMaxB at a time.
static int sample_fullvocab(const void* logits, int R, int V, int dtype, const float* temperature, float top_p,
                            uint64_t seed, int32_t* out_tokens, void* workspace, uint32_t* status, void* stream) {
  const int mode = top_p >= 1.0f ? kModeFullVocab : kModeFullVocabTopP;
  const size_t row_bytes = (size_t)V * esize_of(dtype);
  for (int r0 = 0; r0 < R; r0 += kMaxB) {
    const int n = R - r0 < kMaxB ? R - r0 : kMaxB;
    Params p = base_params(dtype, V);
    p.target = static_cast<const unsigned char*>(logits) + (size_t)r0 * row_bytes;
    p.draft = p.target;  // no draft rows are read (gamma = 0)
    p.draft_tokens = nullptr;
    p.temperature = temperature + r0;
    p.B = n;
    p.gamma = 0;
    p.top_k = 0;
    p.top_p = top_p >= 1.0f ? 1.0f : top_p;
    p.seed = seed;
    p.task = kTaskVerify;
    p.row_base = r0;
    p.out_tokens = out_tokens + r0;
    p.out_len = nullptr;
    p.status = status;
    bind_workspace(p, workspace, n, n, mode);
    const int rc = run_step(p, n, workspace, stream, true);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

static int rows_task(int task, const void* logits, int R, int V, int dtype, const float* temperature, int top_k,
                     float top_p, uint64_t seed, int32_t* out_tokens, int32_t* out_idx, float* out_prob,
                     int32_t* out_count, void* workspace, size_t workspace_bytes, uint32_t* status, void* stream) {
  if (R < 1 || V < 1 || !esize_of(dtype))
    return fail(DFLASH_ERR_INVALID_ARG, "bad shape R=%d V=%d dtype=%d", R, V, dtype);
  if (!logits || !temperature || !workspace) return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  const int mode = filter_mode(V, top_k, top_p);
  if (mode < 0) return fail(DFLASH_ERR_INVALID_ARG, "top_p=%g must be in (0, 1]", (double)top_p);
  if (mode != kModeTopK && !(whole_vocab(mode) && task == kTaskSample))
    return fail(DFLASH_ERR_UNSUPPORTED,
                "top_k=%d with top_p=%g is not supported here (need 1 <= top_k <= %d and top_k < V; the "
                "sampler also takes top-k off)",
                top_k, (double)top_p, DFLASH_MAX_TOP_K);
  int rc = check_aligned(logits, esize_of(dtype), "logits");
  if (rc) return rc;
  const size_t need = dflash_rows_workspace_bytes(R, V, dtype, top_k, top_p);
  if (workspace_bytes < need)
    return fail(DFLASH_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes,
                need);
  if (whole_vocab(mode))
    return sample_fullvocab(logits, R, V, dtype, temperature, top_p, seed, out_tokens, workspace, status, stream);
  Params p = base_params(dtype, V);
  p.temperature = temperature;
  p.gamma = 1;  // unused by the rows tasks (a row is its own slot); any valid value
  p.top_k = top_k;
  p.top_p = top_p >= 1.0f ? 1.0f : top_p;
  p.seed = seed;
  p.task = task;
  p.status = status;
  const int chunk = R < kMaxCounterSlots ? R : kMaxCounterSlots;
  bind_workspace(p, workspace, chunk, 1);
  // rows go through launches of at most kMaxCounterSlots rows each (the size
  // of the workspace's counter header); the sampler keys its uniforms by the
  // absolute row index, so each launch is told where its rows start
  for (int r0 = 0; r0 < R; r0 += chunk) {
    const int n = R - r0 < chunk ? R - r0 : chunk;
    const size_t row_bytes = (size_t)V * esize_of(dtype);
    p.target = static_cast<const unsigned char*>(logits) + (size_t)r0 * row_bytes;
    p.temperature = temperature + r0;
    p.B = n;
    p.row_base = r0;
    p.out_tokens = out_tokens ? out_tokens + r0 : nullptr;
    p.out_idx = out_idx ? out_idx + (size_t)r0 * top_k : nullptr;
    p.out_prob = out_prob ? out_prob + (size_t)r0 * top_k : nullptr;
    p.out_count = out_count ? out_count + r0 : nullptr;
    rc = run(p, n, stream);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

int dflash_filter(const void* logits, int R, int V, int dtype, const float* temperature, int top_k, float top_p,
                  int32_t* out_idx, float* out_prob, int32_t* out_count, void* workspace, size_t workspace_bytes,
                  uint32_t* status, void* stream) {
  NvtxRange nvtx_range("dflash_filter");
  if (!out_idx || !out_prob || !out_count) return fail(DFLASH_ERR_INVALID_ARG, "null output pointer");
  return rows_task(kTaskFilter, logits, R, V, dtype, temperature, top_k, top_p, 0, nullptr, out_idx, out_prob,
                   out_count, workspace, workspace_bytes, status, stream);
}

int dflash_sample(const void* logits, int R, int V, int dtype, const float* temperature, int top_k, float top_p,
                  uint64_t seed, int32_t* out_tokens, void* workspace, size_t workspace_bytes, uint32_t* status,
                  void* stream) {
  NvtxRange nvtx_range("dflash_sample");
  if (!out_tokens) return fail(DFLASH_ERR_INVALID_ARG, "null output pointer");
  return rows_task(kTaskSample, logits, R, V, dtype, temperature, top_k, top_p, seed, out_tokens, nullptr, nullptr,
                   nullptr, workspace, workspace_bytes, status, stream);
}

size_t dflash_candidates_words(int B, int gamma, int k) {
  if (B < 1 || B > kMaxB || gamma < 1 || gamma > kMaxGamma || k < 1 || k > DFLASH_MAX_TOP_K) return 0;
  return candidate_layout(B, gamma, k).words;
}

size_t dflash_shard_workspace_bytes(int B, int gamma, int V_shard, int dtype, int k) {
  if (B < 1 || B > kMaxB || gamma < 1 || gamma > kMaxGamma || k < 1 || k > DFLASH_MAX_TOP_K || k >= V_shard)
    return 0;
  return dflash_rows_workspace_bytes(B * (gamma + 1), V_shard, dtype, k, 1.0f);
}

// one candidates pass over R rows of a vocabulary shard
static int candidates_pass(const void* logits, int R, int V_shard, int dtype, int vocab_offset, int k,
                           float* out_logit, int32_t* out_token, float* out_max, void* workspace, uint32_t* status,
                           void* stream) {
  Params p = base_params(dtype, V_shard);
  p.gamma = 1;  // unused by the rows tasks (a row is its own slot); any valid value
  p.top_k = k;
  p.top_p = 1.0f;
  p.task = kTaskCandidates;
  p.vocab_offset = vocab_offset;
  p.status = status;
  const int chunk = R < kMaxCounterSlots ? R : kMaxCounterSlots;
  bind_workspace(p, workspace, chunk, 1);
  const size_t row_bytes = (size_t)V_shard * esize_of(dtype);
  for (int r0 = 0; r0 < R; r0 += chunk) {
    const int n = R - r0 < chunk ? R - r0 : chunk;
    p.target = static_cast<const unsigned char*>(logits) + (size_t)r0 * row_bytes;
    p.B = n;
    p.row_base = r0;
    p.out_prob = out_logit + (size_t)r0 * k;
    p.out_idx = out_token + (size_t)r0 * k;
    p.out_rowmax = out_max + r0;
    const int rc = run(p, n, stream);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

int dflash_shard_candidates(const void* target_shard, const void* draft_shard, int B, int gamma, int V_shard,
                            int dtype, int vocab_offset, int k, uint32_t* record, void* workspace,
                            size_t workspace_bytes, uint32_t* status, void* stream) {
  NvtxRange nvtx_range("dflash_shard_candidates");
  int rc = check_shape(B, gamma, V_shard, dtype);
  if (rc) return rc;
  if (!target_shard || !draft_shard || !record || !workspace)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  if (k < 1 || k > DFLASH_MAX_TOP_K || k >= V_shard)
    return fail(DFLASH_ERR_INVALID_ARG, "k=%d must be in [1, %d] and below the shard's V=%d", k, DFLASH_MAX_TOP_K,
                V_shard);
  if (vocab_offset < 0 || (long long)vocab_offset + V_shard > 0x7fffffffLL)
    return fail(DFLASH_ERR_INVALID_ARG, "vocab_offset=%d puts the shard's tokens outside [0, 2^31)", vocab_offset);
  const int es = esize_of(dtype);
  if ((rc = check_aligned(target_shard, es, "target_shard")) || (rc = check_aligned(draft_shard, es, "draft_shard")))
    return rc;
  if (((uintptr_t)record) % 4u) return fail(DFLASH_ERR_INVALID_ARG, "record is not 4-byte aligned");
  const size_t need = dflash_shard_workspace_bytes(B, gamma, V_shard, dtype, k);
  if (workspace_bytes < need)
    return fail(DFLASH_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes,
                need);
  const CandidateLayout L = candidate_layout(B, gamma, k);
  float* f = reinterpret_cast<float*>(record);
  int32_t* t = reinterpret_cast<int32_t*>(record);
  rc = candidates_pass(target_shard, B * (gamma + 1), V_shard, dtype, vocab_offset, k, f + L.t_logit, t + L.t_token,
                       f + L.t_max, workspace, status, stream);
  if (rc) return rc;
  return candidates_pass(draft_shard, B * gamma, V_shard, dtype, vocab_offset, k, f + L.d_logit, t + L.d_token,
                         f + L.d_max, workspace, status, stream);
}

int dflash_verify_candidates(const uint32_t* records, int n_shards, int k, const int32_t* draft_tokens, int B,
                             int gamma, int V, const float* temperature, int top_k, float top_p, uint64_t seed,
                             int32_t* out_tokens, int32_t* out_accept_len, uint32_t* status, void* stream) {
  NvtxRange nvtx_range("dflash_verify_candidates");
  if (B < 1 || B > kMaxB) return fail(DFLASH_ERR_INVALID_ARG, "B=%d outside [1, %d]", B, kMaxB);
  if (gamma < 1 || gamma > kMaxGamma)
    return fail(DFLASH_ERR_INVALID_ARG, "gamma=%d outside [1, %d]", gamma, kMaxGamma);
  if (V < 1) return fail(DFLASH_ERR_INVALID_ARG, "V=%d must be >= 1", V);
  if (!records || !draft_tokens || !temperature || !out_tokens || !out_accept_len)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  if (((uintptr_t)records) % 4u) return fail(DFLASH_ERR_INVALID_ARG, "records are not 4-byte aligned");
  if (k < 1 || k > DFLASH_MAX_TOP_K) return fail(DFLASH_ERR_INVALID_ARG, "k=%d outside [1, %d]", k, DFLASH_MAX_TOP_K);
  if (n_shards < 1 || (long long)n_shards * k > kMaxShardCand)
    return fail(DFLASH_ERR_INVALID_ARG, "n_shards=%d with k=%d: need 1 <= n_shards * k <= %d", n_shards, k,
                kMaxShardCand);
  const int mode = filter_mode(V, top_k, top_p);
  if (mode < 0) return fail(DFLASH_ERR_INVALID_ARG, "top_p=%g must be in (0, 1]", (double)top_p);
  if (mode != kModeTopK || top_k > k)
    return fail(DFLASH_ERR_UNSUPPORTED,
                "top_k=%d with top_p=%g is not supported from shard candidates (need 1 <= top_k <= k = %d and "
                "top_k < V)",
                top_k, (double)top_p, k);
  CandParams c;
  memset(&c, 0, sizeof c);
  c.L = candidate_layout(B, gamma, k);
  c.records = records;
  c.words = c.L.words;
  c.n_shards = n_shards;
  c.k = k;
  c.draft_tokens = draft_tokens;
  c.temperature = temperature;
  c.B = B;
  c.gamma = gamma;
  c.V = V;
  c.top_k = top_k;
  c.top_p = top_p >= 1.0f ? 1.0f : top_p;
  c.seed = seed;
  c.out_tokens = out_tokens;
  c.out_len = out_accept_len;
  c.status = status;
  const Exp2Table& et = exp2_table();
  memcpy(c.exp2.hi, et.hi, sizeof et.hi);
  memcpy(c.exp2.lo, et.lo, sizeof et.lo);
  const int e = launch_verify_candidates(c, stream);
  if (e) return cuda_fail((cudaError_t)e, "launching the verification from shard candidates");
  return DFLASH_OK;
}

int dflash_uniforms(uint64_t seed, int B, int npos, int stream_id, float* out_accept, float* out_draw, void* stream) {
  if (B < 1 || npos < 1 || (!out_accept && !out_draw))
    return fail(DFLASH_ERR_INVALID_ARG, "bad uniforms arguments");
  const int e = launch_uniforms(seed, B, npos, stream_id, out_accept, out_draw, stream);
  if (e) return cuda_fail((cudaError_t)e, "launching the uniforms kernel");
  return DFLASH_OK;
}

}  // extern "C"
