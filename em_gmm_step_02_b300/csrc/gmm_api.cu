// gmm_api.cu -- host side of the C ABI declared in include/gmm.h: argument
// checks, the launch plan (precision, cluster size, single or two-pass),
// the per-device workspace, and the launch sequence of one EM step.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "gmm.h"
#include "gmm_kernels.cuh"
#include "layout.cuh"

using namespace gmm;

namespace {

thread_local std::string g_error;
thread_local int32_t g_launches = 0;

// Optional timing of the main (fused) kernel launches: an event pair around
// each, read back by gmm_profile_end().
thread_local bool g_prof_on = false;
thread_local std::vector<std::pair<cudaEvent_t, cudaEvent_t>> g_prof_events;
thread_local int32_t g_prof_launches = 0;

int fail(int code, const std::string& msg) {
  g_error = msg;
  return code;
}

#define CUDA_TRY(expr)                                                                  \
  do {                                                                                  \
    cudaError_t e_ = (expr);                                                            \
    if (e_ != cudaSuccess) return fail(GMM_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString(e_)); \
  } while (0)

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// ------------------------------------------------------------------ plan
struct Plan {
  int64_t N;
  int D, K, cov_diag, x_bf16;
  bool fast;
  int nch, np, nst;
  int K_pad, n_slices;
  int n_tiles;
  bool two_pass;
  int C;              // cluster size of the single pass
  int C1;             // cluster size of the top-m pass (two-pass): 8, or 1 in the SPLIT plan
  int n_kgroups;      // K groups of the top-m pass (two-pass)
  int C1e;            // cluster size of the EM step's normaliser pass (two-pass)
  int n_kgroups_e;    // K groups of the EM step's normaliser pass
  int tg1e;           // tile groups of the EM step's normaliser pass
  int tg;             // tile groups of the statistics pass
  int tg1;            // tile groups of pass 1 (two-pass)
  int F;
  int flush;
  uint32_t max_polls; // polls per device-side wait (0: the kernels' default)
  size_t smem;        // dynamic shared memory of the E-step kernel
  bool emfast;        // the E-step passes run the two-team kernel (em_fast.cu): FAST, two-pass plan
  int threads;        // threads per CTA of the E-step kernel
  // workspace offsets
  size_t off_meta, off_pimg, off_cimg, off_cadj, off_iscale, off_part, off_llpart, off_lsepart, off_lse, off_ll;
  // tied covariance (cov_diag == 2): L, Sigma^-1, solve scratch, log|Sigma|, Gram
  // matrix and its partials, per-component (N_k, nu_k), covariance scratch
  size_t off_tl, off_sinv, off_twork, off_logdet, off_gram, off_gpart, off_tstats, off_tsig;
  int n_gram;
  size_t n_llpart;
  size_t ws_bytes;
};

constexpr int kCombineBlocks = 296;
// default rows per chunk of the host-data entry point (256 MiB of bf16 rows at
// D = 128): the last chunk's kernels are the part of a step that no copy
// overlaps, so smaller chunks bring the step closer to the host link's time
// (10M x 128 bf16: 47.3 ms per step at 2^20 rows, 51.0 ms at 2^22)
constexpr int64_t kHostChunkRows = int64_t(1) << 20;
constexpr size_t kStatusBytes = 256;

int device_sms() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  return sms;
}

}  // namespace

namespace {

template <int NP, int NCH, int NST>
constexpr size_t cfg_smem() {
  return Cfg<NP, NCH, NST>::kEnd + 1024;   // + base alignment slack
}

size_t fused_smem(int np, int nch, int nst) {
  size_t b = 0;
  if (np == 1 && nch == 1 && nst == 2) b = cfg_smem<1, 1, 2>();
  else if (np == 1 && nch == 2 && nst == 2) b = cfg_smem<1, 2, 2>();
  else if (np == 2 && nch == 1 && nst == 1) b = cfg_smem<2, 1, 1>();
  else if (np == 2 && nch == 2 && nst == 1) b = cfg_smem<2, 2, 1>();
  return std::max<size_t>(b, 120 * 1024);   // one CTA per SM: it owns all of tensor memory
}

const void* fused_fn(int np, int nch, int nst, bool topm = false) {
  if (np == 1 && nch == 1 && nst == 2) return kernel_handle(topm ? K_TOPM_1_1_2 : K_FUSED_1_1_2);
  if (np == 1 && nch == 2 && nst == 2) return kernel_handle(topm ? K_TOPM_1_2_2 : K_FUSED_1_2_2);
  if (np == 2 && nch == 1 && nst == 1) return kernel_handle(topm ? K_TOPM_2_1_1 : K_FUSED_2_1_1);
  if (np == 2 && nch == 2 && nst == 1) return kernel_handle(topm ? K_TOPM_2_2_1 : K_FUSED_2_2_1);
  return nullptr;
}

// Largest number of C-CTA clusters of the fused kernel resident at once.
int max_clusters(const void* fn, size_t smem, int C, int threads) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_pair(fn, C);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int sms = device_sms();
  int n = std::max(1, sms / C);
  // the occupancy query needs the kernel's dynamic shared-memory limit raised first
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return n;
  }
  if (C > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C * n, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int got = 0;
    if (cudaOccupancyMaxActiveClusters(&got, fn, &cfg) == cudaSuccess && got > 0) n = got;
    else cudaGetLastError();
  }
  cache[key] = n;
  return n;
}

int make_plan(Plan& p, const void* X, int64_t N, int32_t D, int32_t K, int32_t cov, int32_t dtype,
              const gmm_opts& o, bool need_device) {
  if (N < 1) return fail(GMM_ERR_INVALID_ARG, "N must be >= 1");
  if (D < 1) return fail(GMM_ERR_INVALID_ARG, "D must be >= 1");
  if (K < 1) return fail(GMM_ERR_INVALID_ARG, "K must be >= 1");
  if (cov != GMM_SPHERICAL && cov != GMM_DIAG && cov != GMM_TIED)
    return fail(GMM_ERR_INVALID_ARG, "cov_type must be 0, 1 or 2");
  if (dtype != GMM_F32 && dtype != GMM_BF16) return fail(GMM_ERR_INVALID_ARG, "x_dtype must be 0 or 1");
  if (o.precision < GMM_PREC_AUTO || o.precision > GMM_PREC_PRECISE)
    return fail(GMM_ERR_INVALID_ARG, "unknown precision");
  if (o.plan < GMM_PLAN_AUTO || o.plan > GMM_PLAN_SPLIT) return fail(GMM_ERR_INVALID_ARG, "unknown plan");
  if (o.wait_limit < 0) return fail(GMM_ERR_INVALID_ARG, "wait_limit must be >= 0");
  if (o.topm_refine < GMM_REFINE_AUTO || o.topm_refine > GMM_REFINE_OFF)
    return fail(GMM_ERR_INVALID_ARG, "topm_refine must be 0 (AUTO), 1 (ON) or 2 (OFF)");
  if (!(o.reg_covar >= 0.f) || !(o.var_floor >= 0.f) || !std::isfinite(o.reg_covar) || !std::isfinite(o.var_floor))
    return fail(GMM_ERR_INVALID_ARG, "reg_covar and var_floor must be finite and >= 0");
  if (!(o.x_absmax >= 0.f) || !std::isfinite(o.x_absmax)) return fail(GMM_ERR_INVALID_ARG, "x_absmax must be finite and >= 0");
  if (D > kMaxD) return fail(GMM_ERR_UNSUPPORTED, "D > 128 is not supported");
  if (K > 8192) return fail(GMM_ERR_UNSUPPORTED, "K > 8192 is not supported");
  if (N > (int64_t(1) << 40)) return fail(GMM_ERR_UNSUPPORTED, "N too large");
  if (X && (reinterpret_cast<uintptr_t>(X) & 15)) return fail(GMM_ERR_INVALID_ARG, "X must be 16-byte aligned");
  p.N = N; p.D = D; p.K = K; p.cov_diag = cov; p.x_bf16 = dtype == GMM_BF16;
  p.max_polls = static_cast<uint32_t>(o.wait_limit);
  const int prec = o.precision == GMM_PREC_AUTO ? (p.x_bf16 ? GMM_PREC_FAST : GMM_PREC_PRECISE) : o.precision;
  p.fast = prec == GMM_PREC_FAST;
  p.nch = D <= 64 ? 1 : 2;
  p.np = p.fast ? 1 : 2;
  p.nst = p.fast ? 2 : 1;
  p.n_slices = (K + kSlice - 1) / kSlice;
  const bool split = o.plan == GMM_PLAN_SPLIT;
  p.two_pass = split || p.n_slices > 8;
  p.C1 = split ? 1 : 8;
  if (p.two_pass && !split) p.n_slices = (p.n_slices + 7) / 8 * 8;   // whole 8-slice groups for pass 1
  p.K_pad = p.n_slices * kSlice;
  p.n_tiles = static_cast<int>((N + kBN - 1) / kBN);
  p.emfast = p.fast && p.two_pass;
  p.smem = p.emfast ? emfast_smem(p.nch) : fused_smem(p.np, p.nch, p.nst);
  p.threads = p.emfast ? kEmFastThreads : 416;
  p.F = 2 * p.nch * kAtomElems + 1;
  p.flush = p.fast ? 128 : 16;
  const int sms = need_device ? device_sms() : 148;
  const void* fn = p.emfast ? emfast_handle(p.nch, MODE_LSE) : fused_fn(p.np, p.nch, p.nst);
  if (!p.two_pass) {
    p.C = p.n_slices;
    p.n_kgroups = 1;
    int mc = need_device ? max_clusters(fn, p.smem, p.C, p.threads) : std::max(1, sms / p.C);
    p.tg = std::max(1, std::min(p.n_tiles, mc));
    p.tg1 = 0;
    p.C1e = p.C;
    p.n_kgroups_e = 1;
    p.tg1e = 0;
  } else {
    p.C = p.C1;
    p.n_kgroups = p.n_slices / p.C1;
    int mc = p.C1 == 1 ? sms : (need_device ? max_clusters(fn, p.smem, p.C1, p.threads) : std::max(1, sms / p.C1));
    // every K group gets as many tile groups as clusters can be resident at
    // once; the groups run one after another in waves, each keeping the GPU full
    p.tg1 = std::max(1, std::min(p.n_tiles, mc));
    // The EM step's normaliser pass runs without clusters (one normaliser per
    // slice, no cross-CTA waits, every SM) when the per-slice normalisers fit
    // in 4 GiB; the top-m pass keeps its groups of 8 (its candidate lists grow
    // with the number of K groups).
    const bool split_e = split || (o.plan == GMM_PLAN_AUTO &&
                                   static_cast<double>(N) * p.n_slices * sizeof(float) <= 4.0 * (1 << 30));
    p.C1e = split_e ? 1 : p.C1;
    p.n_kgroups_e = p.n_slices / p.C1e;
    p.tg1e = p.C1e == p.C1 ? p.tg1 : std::max(1, std::min(p.n_tiles, sms));
    // statistics pass: n_slices x tg CTAs, one per SM at a time.  tg is chosen
    // so that the waves come out nearly full (cost = waves x tiles per CTA),
    // with the partial statistics (tg x K_pad x F doubles) at most 256 MiB.
    int best = std::max(1, std::min(p.n_tiles, sms / p.n_slices));
    int64_t best_cost = int64_t(1) << 62;
    for (int tg = 1; tg <= std::min(p.n_tiles, 64); ++tg) {
      if (static_cast<double>(tg) * p.K_pad * p.F * sizeof(double) > 256.0 * (1 << 20)) break;
      const int64_t waves = (static_cast<int64_t>(p.n_slices) * tg + sms - 1) / sms;
      const int64_t cost = waves * ((p.n_tiles + tg - 1) / tg);
      if (cost < best_cost) {
        best_cost = cost;
        best = tg;
      }
    }
    p.tg = best;
  }
  // workspace layout
  size_t off = kStatusBytes;
  p.off_meta = off; off += align256(sizeof(Meta));
  p.off_ll = off; off += 256;
  const size_t piece = static_cast<size_t>(2 * p.nch) * kChunkBytes;
  p.off_pimg = off; off += align256(static_cast<size_t>(p.n_slices) * p.np * piece);
  p.off_cimg = off; off += align256(static_cast<size_t>(p.n_slices) * kConstBytes);
  p.off_cadj = off; off += align256(sizeof(float) * p.K_pad);
  p.off_iscale = off; off += align256(sizeof(float) * p.K_pad);
  p.off_part = off; off += align256(sizeof(double) * static_cast<size_t>(p.tg) * p.K_pad * p.F);
  p.n_llpart = std::max<size_t>(static_cast<size_t>(p.tg) * p.C, kCombineBlocks);
  p.off_llpart = off; off += align256(sizeof(double) * p.n_llpart);
  p.off_lsepart = off;
  p.off_lse = off;
  if (p.two_pass) {
    off += align256(sizeof(float) * static_cast<size_t>(std::max(p.n_kgroups, p.n_kgroups_e)) * N);
    p.off_lse = off;
    off += align256(sizeof(float) * static_cast<size_t>(N));
  }
  p.n_gram = 0;
  p.off_tl = p.off_sinv = p.off_twork = p.off_logdet = p.off_gram = p.off_gpart = p.off_tstats = p.off_tsig = off;
  if (p.cov_diag == GMM_TIED) {
    const size_t dd = sizeof(double) * static_cast<size_t>(D) * D;
    p.n_gram = std::max(1, std::min(p.n_tiles, 2 * sms));   // one partial per CTA of the Gram kernel (two per SM)
    p.off_tl = off; off += align256(dd);
    p.off_sinv = off; off += align256(dd);
    p.off_twork = off; off += align256(dd);
    p.off_logdet = off; off += 256;
    p.off_gram = off; off += align256(dd);
    p.off_gpart = off; off += align256(dd * p.n_gram);
    p.off_tstats = off; off += align256(sizeof(double) * static_cast<size_t>(K) * (D + 1));
    p.off_tsig = off; off += align256(sizeof(float) * static_cast<size_t>(D) * D);
  }
  p.ws_bytes = off;
  return GMM_OK;
}

// ------------------------------------------------------------------ workspace
struct Workspace {
  uint8_t* buf = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mu;
std::map<int, Workspace> g_ws;

int get_workspace(size_t need, uint8_t** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Workspace& w = g_ws[dev];
  if (w.bytes < need) {
    uint32_t old_status = 0;
    if (w.buf) {
      CUDA_TRY(cudaDeviceSynchronize());
      CUDA_TRY(cudaMemcpy(&old_status, w.buf, sizeof(uint32_t), cudaMemcpyDeviceToHost));
      CUDA_TRY(cudaFree(w.buf));
      w.buf = nullptr;
      w.bytes = 0;
    }
    size_t bytes = std::max(need, w.bytes + w.bytes / 2);
    CUDA_TRY(cudaMalloc(&w.buf, bytes));
    CUDA_TRY(cudaMemset(w.buf, 0, kStatusBytes));
    if (old_status) CUDA_TRY(cudaMemcpy(w.buf, &old_status, sizeof(uint32_t), cudaMemcpyHostToDevice));
    w.bytes = bytes;
  }
  *out = w.buf;
  return GMM_OK;
}

int status_to_code(uint32_t st, uint32_t where = 0) {
  if (st & ST_TIMEOUT) {
    char buf[160];
    snprintf(buf, sizeof buf, "a device-side wait exceeded its bound (first: thread %u, barrier at shared offset 0x%x)",
             (where >> 20) & 0x7FFu, where & 0xFFFFFu);
    return fail(GMM_ERR_TIMEOUT, where ? std::string(buf) : std::string("a device-side wait exceeded its bound"));
  }
  if (st & ST_NONFINITE) return fail(GMM_ERR_NONFINITE, "a parameter is not finite or a variance is not positive");
  if (st & ST_RANGE) return fail(GMM_ERR_RANGE, "data magnitude outside the FAST operand range");
  if (st & ST_CAPACITY)
    return fail(GMM_ERR_CAPACITY, "more threshold-assignment entries than the output capacity (count in offsets[N])");
  return GMM_OK;
}

template <typename... Args>
int launch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (cluster > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* argv[] = {static_cast<void*>(&args)...};
  CUDA_TRY(cudaLaunchKernelExC(&cfg, fn, argv));
  ++g_launches;
  return GMM_OK;
}

// Launch of a main kernel, bracketed by events when profiling is on.
template <typename... Args>
int launch_main(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster, Args... args) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (g_prof_on) {
    CUDA_TRY(cudaEventCreate(&e0));
    CUDA_TRY(cudaEventCreate(&e1));
    CUDA_TRY(cudaEventRecord(e0, s));
  }
  int r = launch(fn, grid, block, smem, s, cluster, args...);
  if (r) return r;
  if (g_prof_on) {
    CUDA_TRY(cudaEventRecord(e1, s));
    g_prof_events.emplace_back(e0, e1);
    ++g_prof_launches;
  }
  return GMM_OK;
}

int set_smem_attr(const void* fn, size_t smem) {
  CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
  return GMM_OK;
}

int check_ptr(const void* p, const char* name) {
  if (!p) return fail(GMM_ERR_INVALID_ARG, std::string(name) + " is NULL");
  if (reinterpret_cast<uintptr_t>(p) & 3) return fail(GMM_ERR_INVALID_ARG, std::string(name) + " is not 4-byte aligned");
  return GMM_OK;
}

// prep: scan (optional), meta, parameter images
int run_prep(const Plan& p, const void* X, const float* lw, const float* mu, const float* var,
             const gmm_opts& o, uint8_t* ws, cudaStream_t s) {
  Meta* meta = reinterpret_cast<Meta*>(ws + p.off_meta);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  if (o.x_absmax <= 0.f) {
    CUDA_TRY(cudaMemsetAsync(&meta->absmax_bits, 0, sizeof(uint32_t), s));
    const int64_t n_elems = p.N * p.D;
    const int64_t per_vec = p.x_bf16 ? 8 : 4;
    const int sms = device_sms();
    if (n_elems % per_vec == 0) {
      const int64_t n_vec = n_elems / per_vec;
      int blocks = static_cast<int>(std::min<int64_t>(4 * sms, (n_vec + 255) / 256));
      int r = launch(kernel_handle(K_ABSMAX_VEC), dim3(blocks), dim3(256), 0, s, 1,
                     static_cast<const uint4*>(X), n_vec, p.x_bf16, meta);
      if (r) return r;
    } else {
      int blocks = static_cast<int>(std::min<int64_t>(4 * sms, (n_elems + 255) / 256));
      int r = launch(kernel_handle(K_ABSMAX), dim3(blocks), dim3(256), 0, s, 1, X, n_elems,
                     p.x_bf16, meta);
      if (r) return r;
    }
  }
  {
    // bf16 data in FAST stay unshifted: they are then exact in fp16
    int use_shift = (p.fast && p.x_bf16) ? 0 : 1;
    float hint = o.x_absmax;
    int r = launch(kernel_handle(K_META), dim3(1), dim3(128), 0, s, 1, mu, p.D, p.K, use_shift,
                   hint, meta, status);
    if (r) return r;
  }
  const bool tied = p.cov_diag == GMM_TIED;
  double* sinv = tied ? reinterpret_cast<double*>(ws + p.off_sinv) : nullptr;
  double* logdet = tied ? reinterpret_cast<double*>(ws + p.off_logdet) : nullptr;
  if (tied) {
    // Sigma^-1 and log|Sigma| (one block), then the Gram matrix of the data
    const size_t lbytes = sizeof(double) * static_cast<size_t>(p.D) * (p.D + 1);
    int r = set_smem_attr(kernel_handle(K_TIED_PREP), lbytes);
    if (r) return r;
    r = launch(kernel_handle(K_TIED_PREP), dim3(1), dim3(128), lbytes, s, 1, var, p.D,
               reinterpret_cast<double*>(ws + p.off_tl), logdet, status);
    if (r) return r;
    if ((r = set_smem_attr(kernel_handle(K_TIED_INV), lbytes))) return r;
    r = launch(kernel_handle(K_TIED_INV), dim3(p.D), dim3(128), lbytes, s, 1,
               static_cast<const double*>(reinterpret_cast<double*>(ws + p.off_tl)), p.D, sinv);
    if (r) return r;
    if (X) {
      // G = sum (x - shift)(x - shift)^T on the tensor cores: two CTAs per SM,
      // fp64 partials per CTA, fixed-order reduction
      const void* gfn = gram_handle(p.np, p.nch, p.x_bf16 != 0);
      const size_t gsm = gram_smem(p.np, p.nch);
      if ((r = set_smem_attr(gfn, gsm))) return r;
      double* gpart = reinterpret_cast<double*>(ws + p.off_gpart);
      CUDA_TRY(cudaMemsetAsync(gpart, 0, sizeof(double) * static_cast<size_t>(p.n_gram) * p.D * p.D, s));
      FusedArgs ga = {};
      ga.X = X;
      ga.N = p.N;
      ga.D = p.D;
      ga.x_bf16 = p.x_bf16;
      ga.n_tiles = p.n_tiles;
      ga.flush_tiles = p.flush;
      ga.meta = meta;
      ga.status = status;
      ga.max_polls = p.max_polls;
      if ((r = launch(gfn, dim3(p.n_gram), dim3(gram_threads()), gsm, s, 1, ga, gpart))) return r;
      r = launch(kernel_handle(K_GRAM_REDUCE), dim3((p.D * p.D + 255) / 256), dim3(256), 0, s, 1,
                 static_cast<const double*>(gpart), p.n_gram, p.D, static_cast<const Meta*>(meta),
                 reinterpret_cast<double*>(ws + p.off_gram));
      if (r) return r;
    }
  }
  if (p.fast) {
    // the one parameter scale of FAST needs the largest coefficient first
    int r = launch(kernel_handle(K_BMAX), dim3(p.K), dim3(128), 0, s, 1, mu, var, p.D, p.K, p.cov_diag, meta,
                   static_cast<const double*>(sinv));
    if (r) return r;
  }
  {
    const void* fn = kernel_handle(p.fast ? K_PARAMS_FAST : K_PARAMS_PRECISE);
    int r = launch(fn, dim3(p.K_pad), dim3(128), 0, s, 1, lw, mu, var, p.D, p.K, p.cov_diag, p.nch, meta,
                   ws + p.off_pimg, ws + p.off_cimg, reinterpret_cast<float*>(ws + p.off_cadj),
                   reinterpret_cast<float*>(ws + p.off_iscale), status, static_cast<const double*>(sinv),
                   static_cast<const double*>(logdet));
    if (r) return r;
  }
  return GMM_OK;
}

// Tied covariance, after the log-likelihood partials are summed into ll_dev:
// the shared covariance of the M-step into new_vars (when not NULL; else into
// scratch) and the per-point term -1/2 tr(Sigma^-1 G) into ll_dev.
int run_tied_tail(const Plan& p, int K_stats, const gmm_opts& o, uint8_t* ws, float* new_vars, double* ll_dev,
                  cudaStream_t s) {
  float* out = new_vars ? new_vars : reinterpret_cast<float*>(ws + p.off_tsig);
  return launch(kernel_handle(K_SIGMA_TIED), dim3((p.D + 15) / 16, (p.D + 15) / 16), dim3(256), 0, s, 1,
                static_cast<const double*>(reinterpret_cast<double*>(ws + p.off_gram)),
                static_cast<const double*>(reinterpret_cast<double*>(ws + p.off_tstats)), K_stats, p.D, p.N,
                o.reg_covar, o.var_floor, static_cast<const double*>(reinterpret_cast<double*>(ws + p.off_sinv)),
                ll_dev, out);
}

FusedArgs base_args(const Plan& p, const void* X, uint8_t* ws) {
  FusedArgs a = {};
  a.X = X;
  a.N = p.N;
  a.D = p.D;
  a.K = p.K;
  a.K_pad = p.K_pad;
  a.x_bf16 = p.x_bf16;
  a.n_tiles = p.n_tiles;
  a.flush_tiles = p.flush;
  a.F = p.F;
  a.p_img = ws + p.off_pimg;
  a.c_img = ws + p.off_cimg;
  a.cadj = reinterpret_cast<const float*>(ws + p.off_cadj);
  a.iscale = reinterpret_cast<const float*>(ws + p.off_iscale);
  a.meta = reinterpret_cast<const Meta*>(ws + p.off_meta);
  a.part = reinterpret_cast<double*>(ws + p.off_part);
  a.ll_part = reinterpret_cast<double*>(ws + p.off_llpart);
  a.lse_part = reinterpret_cast<float*>(ws + p.off_lsepart);
  a.lse_in = reinterpret_cast<const float*>(ws + p.off_lse);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.max_polls = p.max_polls;
  return a;
}

// E-step kernels over the rows a.X[0, p.N): the fused kernel (one pass), or
// normaliser pass + combine + statistics pass.  The statistics add into the
// partials at a.part (zeroed by the caller once per EM step); the
// log-likelihood partials go to ll_part, *n_ll of them.
// The E-step kernel of a plan (the two-team kernel for FAST).
const void* estep_fn(const Plan& p, int mode) {
  return p.emfast ? emfast_handle(p.nch, mode) : fused_fn(p.np, p.nch, p.nst);
}

// Raise the shared-memory limit of every E-step kernel the plan launches.
int set_estep_attrs(const Plan& p) {
  int r;
  if (!p.two_pass) return set_smem_attr(estep_fn(p, MODE_EM), p.smem);
  if ((r = set_smem_attr(estep_fn(p, MODE_LSE), p.smem))) return r;
  return set_smem_attr(estep_fn(p, MODE_GIVEN), p.smem);
}

int run_estep(const Plan& p, const FusedArgs& a, uint8_t* ws, double* ll_part, cudaStream_t s, int* n_ll) {
  int r;
  if (!p.two_pass) {
    FusedArgs a0 = a;
    a0.mode = MODE_EM;
    a0.C = p.C;
    a0.ll_part = ll_part;
    if ((r = launch_main(estep_fn(p, MODE_EM), dim3(p.C * p.tg, 1), dim3(p.threads), p.smem, s, p.C, a0))) return r;
    *n_ll = p.tg * p.C;   // one log-likelihood partial per CTA
  } else {
    // pass 1: per-point normaliser over each group of 1024 components
    FusedArgs a1 = a;
    a1.mode = MODE_LSE;
    a1.C = p.C1e;
    // without clusters the two-team kernel takes a slice-major grid (the CTAs
    // that run together share their point tiles in L2)
    const dim3 g1 = (p.emfast && p.C1e == 1) ? dim3(p.n_kgroups_e, p.tg1e) : dim3(p.C1e * p.tg1e, p.n_kgroups_e);
    if ((r = launch_main(estep_fn(p, MODE_LSE), g1, dim3(p.threads), p.smem, s, p.C1e, a1))) return r;
    float* lse = reinterpret_cast<float*>(ws + p.off_lse);
    if ((r = launch(kernel_handle(K_LSE_COMBINE), dim3(kCombineBlocks), dim3(256), 0, s, 1,
                    static_cast<const float*>(a.lse_part), p.n_kgroups_e, p.N, lse, ll_part)))
      return r;
    *n_ll = kCombineBlocks;
    // pass 2: statistics of every slice given the normaliser
    FusedArgs a2 = a;
    a2.mode = MODE_GIVEN;
    a2.C = 1;
    a2.ll_part = nullptr;
    if ((r = launch_main(estep_fn(p, MODE_GIVEN), dim3(p.n_slices, p.tg), dim3(p.threads), p.smem, s, 1, a2))) return r;
  }
  return GMM_OK;
}

// M-step from the partials of N_total points, and the total log-likelihood
// (device pointer ll_dev); with loglik_on_host, the copy to the host, the
// wait for the stream and the device status.
int run_finalize(const Plan& p, int64_t N_total, uint8_t* ws, const double* ll_part, int n_ll,
                 const gmm_opts& o, const float* means, const float* vars, float* new_log_weights,
                 float* new_means, float* new_vars, double* total_loglik, cudaStream_t s) {
  double* ll_dev = o.loglik_on_host ? reinterpret_cast<double*>(ws + p.off_ll) : total_loglik;
  float reg = o.reg_covar, floor_ = o.var_floor;
  int Dp = p.nch * kAtomElems;
  int r = launch(kernel_handle(K_FINALIZE), dim3(p.K), dim3(128), 0, s, 1,
                 static_cast<const double*>(reinterpret_cast<double*>(ws + p.off_part)), p.tg, p.K_pad, p.F, Dp,
                 p.D, p.K, N_total, p.cov_diag, reg, floor_,
                 static_cast<double>(p.fast ? kRScale<1>() : kRScale<2>()),
                 static_cast<const Meta*>(reinterpret_cast<Meta*>(ws + p.off_meta)), ll_part, n_ll,
                 new_log_weights, new_means, new_vars, means, vars, ll_dev,
                 p.cov_diag == GMM_TIED ? reinterpret_cast<double*>(ws + p.off_tstats) : nullptr);
  if (r) return r;
  if (p.cov_diag == GMM_TIED && (r = run_tied_tail(p, p.K, o, ws, new_vars, ll_dev, s))) return r;
  if (o.loglik_on_host) {
    CUDA_TRY(cudaMemcpyAsync(total_loglik, ll_dev, sizeof(double), cudaMemcpyDeviceToHost, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    uint32_t st[2] = {0, 0};
    CUDA_TRY(cudaMemcpy(st, ws, sizeof(st), cudaMemcpyDeviceToHost));
    if (st[0]) {
      CUDA_TRY(cudaMemset(ws, 0, sizeof(st)));
      return status_to_code(st[0], st[1]);
    }
  }
  return GMM_OK;
}

// Copy stream and events of the host-data entry point, one set per device.
struct HostPipe {
  cudaStream_t copy = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t copied[2] = {nullptr, nullptr};
  cudaEvent_t freed[2] = {nullptr, nullptr};
};
std::mutex g_pipe_mu;
std::map<int, HostPipe> g_pipes;

int get_pipe(HostPipe** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe& hp = g_pipes[dev];
  if (!hp.copy) {
    CUDA_TRY(cudaStreamCreateWithFlags(&hp.copy, cudaStreamNonBlocking));
    CUDA_TRY(cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming));
    for (int b = 0; b < 2; ++b) {
      CUDA_TRY(cudaEventCreateWithFlags(&hp.copied[b], cudaEventDisableTiming));
      CUDA_TRY(cudaEventCreateWithFlags(&hp.freed[b], cudaEventDisableTiming));
    }
  }
  *out = &hp;
  return GMM_OK;
}

// Wait for the stream and return (and clear) the device status.
int sync_status(uint8_t* ws, cudaStream_t s) {
  CUDA_TRY(cudaStreamSynchronize(s));
  uint32_t st[2] = {0, 0};
  CUDA_TRY(cudaMemcpy(st, ws, sizeof(st), cudaMemcpyDeviceToHost));
  if (st[0]) {
    CUDA_TRY(cudaMemset(ws, 0, sizeof(st)));
    return status_to_code(st[0], st[1]);
  }
  return GMM_OK;
}

// Blocks of the refinement kernel (256 threads, four points per warp): as many
// as are resident at once, at most kRefineMaxBlocks (its log-likelihood partials).
constexpr int kRefineMaxBlocks = 4096;

// Workspace of the top-m pass placed from byte `base` on: per-group
// candidate lists of the K > 1024 plan, then (spherical and diagonal
// covariance) the refinement's per-component rows (mu, 1/s2) padded to kMaxD
// features, its constants (K) and its log-likelihood partials.
struct TopmSpace {
  size_t off_gval, off_gidx, off_ivar, off_cdir, off_rll, end;
};
TopmSpace topm_space(const Plan& p, int m, size_t base) {
  TopmSpace t{base, base, base, base, base, base};
  if (p.two_pass) {
    const size_t lb = align256(sizeof(float) * static_cast<size_t>(p.n_kgroups) * p.N * m);
    t.off_gidx = base + lb;
    t.end = t.off_gidx + lb;
  }
  if (p.cov_diag != GMM_TIED) {
    t.off_ivar = t.end;
    t.off_cdir = t.off_ivar + align256(2 * sizeof(float) * static_cast<size_t>(p.K) * kMaxD);
    t.off_rll = t.off_cdir + align256(sizeof(float) * p.K);
    t.end = t.off_rll + align256(sizeof(double) * kRefineMaxBlocks);
  }
  return t;
}

// FAST top-m runs on the two-team kernel when its candidate lists fit the
// R area: lists of at most 8 and a cluster size that divides the 128 rows.
bool topm_two_team(const Plan& p, int m) {
  const int C = p.two_pass ? p.C1 : p.C;
  return p.fast && m <= 8 && (C == 1 || C == 2 || C == 4 || C == 8);
}

const void* topm_fn(const Plan& p, int m) {
  const int maxm = m <= 2 ? 2 : m <= 4 ? 4 : m <= 8 ? 8 : 16;
  return topm_two_team(p, m) ? emfast_handle(p.nch, MODE_TOPM, maxm) : fused_fn(p.np, p.nch, p.nst, true);
}

size_t topm_smem(const Plan& p, int m) {
  return topm_two_team(p, m) ? emfast_smem(p.nch) : fused_smem(p.np, p.nch, p.nst);
}

// The top-m pass over X: each point's m largest responsibilities and their
// components into resp_out / idx_out (N x m, device); the total
// log-likelihood into ll_dev when it is not NULL.  When refinement is on
// (refine_mode: gmm_refine_t; AUTO = PRECISE only) and the covariance is
// spherical or diagonal, the pass's candidates are then refined from the
// direct form of the log-density (topm_refine.cu: responsibilities, order
// and log-likelihood) using the parameters as given.
int run_topm(const Plan& p, const void* X, int m, float* resp_out, int32_t* idx_out, double* ll_dev, uint8_t* ws,
             const TopmSpace& ts, cudaStream_t s, const float* log_weights, const float* means,
             const float* vars, int refine_mode) {
  const bool refine = p.cov_diag != GMM_TIED && p.N > 0 &&
                      (refine_mode == GMM_REFINE_ON || (refine_mode == GMM_REFINE_AUTO && !p.fast));
  double* ll_pass = refine ? nullptr : ll_dev;
  const int maxm = m <= 2 ? 2 : m <= 4 ? 4 : m <= 8 ? 8 : 16;
  const int C = p.two_pass ? p.C1 : p.C;
  const bool team = topm_two_team(p, m);
  const void* fn = team ? emfast_handle(p.nch, MODE_TOPM, maxm) : fused_fn(p.np, p.nch, p.nst, true);
  const size_t smem = team ? emfast_smem(p.nch) : fused_smem(p.np, p.nch, p.nst);
  const int threads = team ? kEmFastThreads : 416;
  (void)C;
  FusedArgs a = base_args(p, X, ws);
  a.mode = MODE_TOPM;
  a.topm = m;
  a.topm_max = maxm;
  int r;
  // (the candidate lists live in the idle data stage / R area)
  if (!p.two_pass) {
    a.C = p.C;
    a.topm_groups = 1;
    a.topm_val = resp_out;
    a.topm_idx = idx_out;
    if ((r = launch_main(fn, dim3(p.C * p.tg, 1), dim3(threads), smem, s, p.C, a))) return r;
    if (ll_pass && (r = launch(kernel_handle(K_LL_TOTAL), dim3(1), dim3(32), 0, s, 1,
                               static_cast<const double*>(a.ll_part), p.tg * p.C, ll_pass)))
      return r;
  } else {
    a.C = p.C1;
    a.topm_groups = p.n_kgroups;
    a.topm_val = reinterpret_cast<float*>(ws + ts.off_gval);
    a.topm_idx = reinterpret_cast<int32_t*>(ws + ts.off_gidx);
    if ((r = launch_main(fn, dim3(p.C1 * p.tg1, p.n_kgroups), dim3(threads), smem, s, p.C1, a))) return r;
    if ((r = launch(kernel_handle(K_TOPM_COMBINE), dim3(kCombineBlocks), dim3(256), 0, s, 1,
                    static_cast<const float*>(a.lse_part), static_cast<const float*>(a.topm_val),
                    static_cast<const int32_t*>(a.topm_idx), p.n_kgroups, p.N, m, resp_out, idx_out,
                    a.ll_part)))
      return r;
    if (ll_pass && (r = launch(kernel_handle(K_LL_TOTAL), dim3(1), dim3(32), 0, s, 1,
                               static_cast<const double*>(a.ll_part), kCombineBlocks, ll_pass)))
      return r;
  }
  if (refine) {
    float2* pm = reinterpret_cast<float2*>(ws + ts.off_ivar);
    float* cdir = reinterpret_cast<float*>(ws + ts.off_cdir);
    double* rll = ll_dev ? reinterpret_cast<double*>(ws + ts.off_rll) : nullptr;
    // 32 points per block; as many blocks as are resident at once
    const bool vec = p.D % 2 == 0 && (reinterpret_cast<uintptr_t>(X) & (p.x_bf16 ? 3 : 7)) == 0;
    const void* rfn = refine_handle(p.x_bf16 != 0, vec, maxm);
    int per_sm = 2;
    CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rfn, 256, 0));
    const int64_t want = (p.N + 31) / 32;
    const int nblk = static_cast<int>(
        std::min<int64_t>(want, std::min(std::max(per_sm, 1) * device_sms(), kRefineMaxBlocks)));
    if ((r = launch(refine_params_handle(), dim3(p.K), dim3(kMaxD), 0, s, 1, log_weights, means, vars, p.D,
                    p.cov_diag, pm, cdir)))
      return r;
    if ((r = launch(rfn, dim3(nblk), dim3(256), 0, s, 1, X, p.N, p.D, p.K, m,
                    reinterpret_cast<const float4*>(pm), static_cast<const float*>(cdir), resp_out, idx_out, rll)))
      return r;
    if (ll_dev && (r = launch(kernel_handle(K_LL_TOTAL), dim3(1), dim3(32), 0, s, 1, static_cast<const double*>(rll),
                              nblk, ll_dev)))
      return r;
  }
  if (ll_dev && p.cov_diag == GMM_TIED) {
    // the logits' dropped per-point term, from the Gram matrix
    gmm_opts d;
    gmm_default_opts(&d);
    if ((r = run_tied_tail(p, 0, d, ws, nullptr, ll_dev, s))) return r;
  }
  return GMM_OK;
}

// Approximate top-k EM: workspace placed from byte `base` on -- the top-k
// lists (responsibilities, components) of every point, the counting sort's
// per-(tile, component) counts, per-component totals and offsets, the sorted
// pairs, the per-chunk partial statistics and N_k, then the top-m pass's
// own space.
struct TopkSpace {
  int tile;             // points per tile of the counting sort
  int64_t T;            // tiles
  int64_t max_chunks;   // bound on the chunks of kTkChunk pairs over all components
  size_t off_r, off_i, off_cnt, off_tot, off_base, off_cbase, off_pt, off_rw, off_part;
  TopmSpace tm;
  size_t end;
};
TopkSpace topk_space(const Plan& p, int k, size_t base) {
  TopkSpace t;
  const size_t nk = static_cast<size_t>(p.N) * k;
  // 4096 points per tile (the walks count in shared memory), doubled while the
  // count table tiles x K would exceed 2^25 entries
  t.tile = 4096;
  while (static_cast<int64_t>(p.K) * ((p.N + t.tile - 1) / t.tile) > (int64_t(1) << 25)) t.tile *= 2;
  t.T = (p.N + t.tile - 1) / t.tile;
  t.max_chunks = static_cast<int64_t>(nk / kTkChunk) + p.K + 1;
  t.off_r = base;
  t.off_i = t.off_r + align256(sizeof(float) * nk);
  t.off_cnt = t.off_i + align256(sizeof(int32_t) * nk);
  t.off_tot = t.off_cnt + align256(sizeof(int32_t) * static_cast<size_t>(p.K) * t.T);
  t.off_base = t.off_tot + align256(sizeof(int32_t) * p.K);
  t.off_cbase = t.off_base + align256(sizeof(int64_t) * (p.K + 1));
  t.off_pt = t.off_cbase + align256(sizeof(int32_t) * (p.K + 1));
  t.off_rw = t.off_pt + align256(sizeof(uint32_t) * nk);
  t.off_part = t.off_rw + align256(sizeof(float) * nk);
  t.tm = topm_space(p, k, t.off_part + align256(sizeof(double) * static_cast<size_t>(t.max_chunks) * (3 * p.D + 1)));
  t.end = t.tm.end;
  return t;
}

bool approx_topk_on(const gmm_opts& o, int K) { return o.approx_top_k > 0 && o.approx_top_k < K; }

int check_approx_topk(const gmm_opts& o, int64_t N, int K, int cov) {
  if (o.approx_top_k < 0) return fail(GMM_ERR_INVALID_ARG, "approx_top_k must be >= 0");
  if (!approx_topk_on(o, K)) return GMM_OK;
  if (o.approx_top_k > 16) return fail(GMM_ERR_UNSUPPORTED, "approx_top_k must be <= 16 (or >= K for exact EM)");
  if (cov != GMM_SPHERICAL && cov != GMM_DIAG)
    return fail(GMM_ERR_UNSUPPORTED, "approx_top_k needs a spherical or diagonal covariance");
  if (N > 0x7fffffffLL) return fail(GMM_ERR_UNSUPPORTED, "approx_top_k needs N < 2^31");
  return GMM_OK;
}

// The M-step of approximate top-k EM from the top-k lists in the workspace
// (the E-step, run_topm with m = k, has written them).
int run_topk_mstep(const Plan& p, const void* X, int k, const gmm_opts& o, uint8_t* ws, const TopkSpace& t,
                   const float* means, const float* vars, float* new_log_weights, float* new_means, float* new_vars,
                   cudaStream_t s) {
  int r;
  const bool xb = p.x_bf16 != 0;
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + t.off_cnt);
  int32_t* tot = reinterpret_cast<int32_t*>(ws + t.off_tot);
  int64_t* base = reinterpret_cast<int64_t*>(ws + t.off_base);
  int32_t* cbase = reinterpret_cast<int32_t*>(ws + t.off_cbase);
  uint32_t* pt = reinterpret_cast<uint32_t*>(ws + t.off_pt);
  float* rw = reinterpret_cast<float*>(ws + t.off_rw);
  double* part = reinterpret_cast<double*>(ws + t.off_part);
  const int32_t* idx = reinterpret_cast<const int32_t*>(ws + t.off_i);
  const float* resp = reinterpret_cast<const float*>(ws + t.off_r);
  const unsigned tile_blocks = static_cast<unsigned>(t.T);
  const size_t table_bytes = sizeof(int32_t) * static_cast<size_t>(p.K);
  if ((r = set_smem_attr(topk_handle(TK_COUNT, xb), table_bytes))) return r;
  if ((r = set_smem_attr(topk_handle(TK_FILL, xb), table_bytes))) return r;
  const unsigned chunk_blocks = static_cast<unsigned>(t.max_chunks);
  if ((r = launch(topk_handle(TK_COUNT, xb), dim3(tile_blocks), dim3(32), table_bytes, s, 1, idx, p.N, k, p.K, t.T,
                  t.tile, cnt)))
    return r;
  if ((r = launch(topk_handle(TK_SCAN, xb), dim3((p.K + 31) / 32), dim3(1024), 0, s, 1, cnt, p.K, t.T, tot))) return r;
  if ((r = launch(topk_handle(TK_BASE, xb), dim3(1), dim3(1024), 0, s, 1, static_cast<const int32_t*>(tot), p.K,
                  base, cbase)))
    return r;
  if ((r = launch(topk_handle(TK_FILL, xb), dim3(tile_blocks), dim3(32), table_bytes, s, 1, idx, resp, p.N, k, p.K,
                  t.T, t.tile, static_cast<const int32_t*>(cnt), static_cast<const int64_t*>(base), pt, rw)))
    return r;
  // 16-byte row loads when a row is a whole number of 16-byte units
  const bool vec = (p.D * (xb ? 2 : 4)) % 16 == 0;
  if ((r = launch(topk_handle(vec ? TK_STATS_VEC : TK_STATS, xb), dim3(chunk_blocks), dim3(128), 0, s, 1, X, p.D, p.K,
                  static_cast<const int64_t*>(base), static_cast<const int32_t*>(cbase),
                  static_cast<const uint32_t*>(pt), static_cast<const float*>(rw), part)))
    return r;
  return launch(topk_handle(TK_FINAL, xb), dim3(p.K), dim3(128), 0, s, 1, static_cast<const double*>(part),
                static_cast<const int32_t*>(cbase), p.N, p.D, p.cov_diag, o.reg_covar, o.var_floor, means, vars,
                new_log_weights, new_means, new_vars);
}

}  // namespace

// ====================================================================== ABI
extern "C" {

void gmm_default_opts(gmm_opts* o) {
  if (!o) return;
  o->precision = GMM_PREC_AUTO;
  o->reg_covar = 1e-6f;
  o->var_floor = 0.f;
  o->x_absmax = 0.f;
  o->loglik_on_host = 0;
  o->plan = GMM_PLAN_AUTO;
  o->wait_limit = 0;
  o->approx_top_k = 0;
  o->topm_refine = GMM_REFINE_AUTO;
}

const char* gmm_last_error(void) { return g_error.c_str(); }

int32_t gmm_last_launch_count(void) { return g_launches; }

size_t gmm_workspace_bytes(int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype,
                           const gmm_opts* opts) {
  gmm_opts o;
  gmm_default_opts(&o);
  if (opts) o = *opts;
  Plan p;
  int dev_count = 0;
  bool have_dev = cudaGetDeviceCount(&dev_count) == cudaSuccess && dev_count > 0;
  if (!have_dev) cudaGetLastError();
  if (make_plan(p, nullptr, N, D, K, cov_type, x_dtype, o, have_dev) != GMM_OK) return 0;
  if (check_approx_topk(o, N, K, cov_type) != GMM_OK) return 0;
  if (approx_topk_on(o, K)) return topk_space(p, o.approx_top_k, p.ws_bytes).end;
  return p.ws_bytes;
}

int gmm_reserve(int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype, const gmm_opts* opts) {
  gmm_opts o;
  gmm_default_opts(&o);
  if (opts) o = *opts;
  Plan p;
  int r = make_plan(p, nullptr, N, D, K, cov_type, x_dtype, o, true);
  if (r) return r;
  if ((r = check_approx_topk(o, N, K, cov_type))) return r;
  uint8_t* ws = nullptr;
  return get_workspace(approx_topk_on(o, K) ? topk_space(p, o.approx_top_k, p.ws_bytes).end : p.ws_bytes, &ws);
}

int gmm_em_step(const void* X, int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype,
                const float* log_weights, const float* means, const float* vars, float* new_log_weights,
                float* new_means, float* new_vars, double* total_loglik, const gmm_opts* opts, void* stream) {
  g_launches = 0;
  gmm_opts o;
  gmm_default_opts(&o);
  if (opts) o = *opts;
  if (!X) return fail(GMM_ERR_INVALID_ARG, "X is NULL");
  int r;
  if ((r = check_ptr(log_weights, "log_weights")) || (r = check_ptr(means, "means")) ||
      (r = check_ptr(vars, "vars")) || (r = check_ptr(new_log_weights, "new_log_weights")) ||
      (r = check_ptr(new_means, "new_means")) || (r = check_ptr(new_vars, "new_vars")))
    return r;
  if (!total_loglik) return fail(GMM_ERR_INVALID_ARG, "total_loglik is NULL");
  if ((r = check_approx_topk(o, N, K, cov_type))) return r;
  Plan p;
  if ((r = make_plan(p, X, N, D, K, cov_type, x_dtype, o, true))) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = nullptr;
  if (approx_topk_on(o, K)) {
    // approximate top-k EM: the top-m pass (m = k) into the workspace, then
    // the sparse M-step
    const int k = o.approx_top_k;
    const TopkSpace t = topk_space(p, k, p.ws_bytes);
    if ((r = get_workspace(t.end, &ws))) return r;
    if ((r = set_smem_attr(topm_fn(p, k), topm_smem(p, k)))) return r;
    if ((r = run_prep(p, X, log_weights, means, vars, o, ws, s))) return r;
    double* ll_dev = o.loglik_on_host ? reinterpret_cast<double*>(ws + p.off_ll) : total_loglik;
    if ((r = run_topm(p, X, k, reinterpret_cast<float*>(ws + t.off_r), reinterpret_cast<int32_t*>(ws + t.off_i),
                      ll_dev, ws, t.tm, s, log_weights, means, vars, o.topm_refine)))
      return r;
    if ((r = run_topk_mstep(p, X, k, o, ws, t, means, vars, new_log_weights, new_means, new_vars, s))) return r;
    if (o.loglik_on_host) {
      CUDA_TRY(cudaMemcpyAsync(total_loglik, ll_dev, sizeof(double), cudaMemcpyDeviceToHost, s));
      return sync_status(ws, s);
    }
    return GMM_OK;
  }
  if ((r = get_workspace(p.ws_bytes, &ws))) return r;
  if ((r = set_estep_attrs(p))) return r;

  if ((r = run_prep(p, X, log_weights, means, vars, o, ws, s))) return r;
  CUDA_TRY(cudaMemsetAsync(ws + p.off_part, 0, sizeof(double) * static_cast<size_t>(p.tg) * p.K_pad * p.F, s));

  FusedArgs a = base_args(p, X, ws);
  double* ll_part = reinterpret_cast<double*>(ws + p.off_llpart);
  int n_ll = 0;
  if ((r = run_estep(p, a, ws, ll_part, s, &n_ll))) return r;
  return run_finalize(p, p.N, ws, ll_part, n_ll, o, means, vars, new_log_weights, new_means, new_vars,
                      total_loglik, s);
}

int gmm_em_step_host(const void* X_host, int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype,
                     const float* log_weights, const float* means, const float* vars, float* new_log_weights,
                     float* new_means, float* new_vars, double* total_loglik, int64_t chunk_rows,
                     const gmm_opts* opts, void* stream) {
  g_launches = 0;
  gmm_opts o;
  gmm_default_opts(&o);
  if (opts) o = *opts;
  if (!X_host) return fail(GMM_ERR_INVALID_ARG, "X_host is NULL");
  if (!(o.x_absmax > 0.f))
    return fail(GMM_ERR_INVALID_ARG, "gmm_em_step_host needs opts->x_absmax > 0 (a bound on max |X|)");
  if (o.approx_top_k != 0 && o.approx_top_k < K)
    return fail(GMM_ERR_UNSUPPORTED, "gmm_em_step_host runs exact EM only (approx_top_k must be 0 or >= K)");
  if (cov_type == GMM_TIED) return fail(GMM_ERR_UNSUPPORTED, "gmm_em_step_host supports spherical and diagonal covariance");
  if (N < 1) return fail(GMM_ERR_INVALID_ARG, "N must be >= 1");
  if (chunk_rows < 0) return fail(GMM_ERR_INVALID_ARG, "chunk_rows must be >= 0");
  int r;
  if ((r = check_ptr(log_weights, "log_weights")) || (r = check_ptr(means, "means")) ||
      (r = check_ptr(vars, "vars")) || (r = check_ptr(new_log_weights, "new_log_weights")) ||
      (r = check_ptr(new_means, "new_means")) || (r = check_ptr(new_vars, "new_vars")))
    return r;
  if (!total_loglik) return fail(GMM_ERR_INVALID_ARG, "total_loglik is NULL");
  if (chunk_rows == 0) chunk_rows = kHostChunkRows;
  // whole tiles per chunk, so that every chunk's rows start a tile
  chunk_rows = std::max<int64_t>(kBN, chunk_rows / kBN * kBN);
  const int64_t rows = std::min(chunk_rows, N);
  const int64_t n_chunks = (N + rows - 1) / rows;
  Plan p;   // planned for one chunk; the M-step uses all N rows
  if ((r = make_plan(p, nullptr, rows, D, K, cov_type, x_dtype, o, true))) return r;
  const size_t row_bytes = static_cast<size_t>(D) * (p.x_bf16 ? 2 : 4);
  const size_t stage_bytes = align256(static_cast<size_t>(rows) * row_bytes);
  const int n_ll_chunk = p.two_pass ? kCombineBlocks : p.tg * p.C;
  const size_t off_ll_all = p.ws_bytes;
  const size_t off_stage = off_ll_all + align256(sizeof(double) * static_cast<size_t>(n_chunks) * n_ll_chunk);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = nullptr;
  if ((r = get_workspace(off_stage + 2 * stage_bytes, &ws))) return r;
  HostPipe* hp = nullptr;
  if ((r = get_pipe(&hp))) return r;
  if ((r = set_estep_attrs(p))) return r;

  // the copies may overwrite the staging buffers only once the work already
  // on the stream (an earlier call's kernels) is done
  CUDA_TRY(cudaEventRecord(hp->start, s));
  CUDA_TRY(cudaStreamWaitEvent(hp->copy, hp->start, 0));
  if ((r = run_prep(p, nullptr, log_weights, means, vars, o, ws, s))) return r;
  CUDA_TRY(cudaMemsetAsync(ws + p.off_part, 0, sizeof(double) * static_cast<size_t>(p.tg) * p.K_pad * p.F, s));
  double* ll_all = reinterpret_cast<double*>(ws + off_ll_all);
  CUDA_TRY(cudaMemsetAsync(ll_all, 0, sizeof(double) * static_cast<size_t>(n_chunks) * n_ll_chunk, s));
  const uint8_t* src = static_cast<const uint8_t*>(X_host);
  for (int64_t c = 0; c < n_chunks; ++c) {
    const int b = static_cast<int>(c & 1);
    const int64_t r0 = c * rows;
    const int64_t nc = std::min(rows, N - r0);
    uint8_t* stage = ws + off_stage + b * stage_bytes;
    // chunk c reuses the buffer of chunk c - 2 once its kernels are done
    if (c >= 2) CUDA_TRY(cudaStreamWaitEvent(hp->copy, hp->freed[b], 0));
    CUDA_TRY(cudaMemcpyAsync(stage, src + static_cast<size_t>(r0) * row_bytes, static_cast<size_t>(nc) * row_bytes,
                             cudaMemcpyHostToDevice, hp->copy));
    CUDA_TRY(cudaEventRecord(hp->copied[b], hp->copy));
    CUDA_TRY(cudaStreamWaitEvent(s, hp->copied[b], 0));
    Plan pc = p;
    pc.N = nc;
    pc.n_tiles = static_cast<int>((nc + kBN - 1) / kBN);
    FusedArgs a = base_args(pc, stage, ws);
    int n_ll = 0;
    if ((r = run_estep(pc, a, ws, ll_all + c * n_ll_chunk, s, &n_ll))) return r;
    CUDA_TRY(cudaEventRecord(hp->freed[b], s));
  }
  return run_finalize(p, N, ws, ll_all, static_cast<int>(n_chunks * n_ll_chunk), o, means, vars, new_log_weights,
                      new_means, new_vars, total_loglik, s);
}

int gmm_predict_topm(const void* X, int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype,
                     const float* log_weights, const float* means, const float* vars, int32_t m, float* resp_out,
                     int32_t* idx_out, double* total_loglik, const gmm_opts* opts, void* stream) {
  g_launches = 0;
  gmm_opts o;
  gmm_default_opts(&o);
  if (opts) o = *opts;
  if (!X) return fail(GMM_ERR_INVALID_ARG, "X is NULL");
  int r;
  if ((r = check_ptr(log_weights, "log_weights")) || (r = check_ptr(means, "means")) ||
      (r = check_ptr(vars, "vars")) || (r = check_ptr(resp_out, "resp_out")) || (r = check_ptr(idx_out, "idx_out")))
    return r;
  if (o.loglik_on_host && !total_loglik) return fail(GMM_ERR_INVALID_ARG, "loglik_on_host needs total_loglik");
  if (m < 1 || m > 16) return fail(GMM_ERR_UNSUPPORTED, "m must be in [1, 16]");
  if (m > K) return fail(GMM_ERR_INVALID_ARG, "m must not exceed K");
  Plan p;
  if ((r = make_plan(p, X, N, D, K, cov_type, x_dtype, o, true))) return r;
  TopmSpace ts = topm_space(p, m, p.ws_bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = nullptr;
  if ((r = get_workspace(ts.end, &ws))) return r;
  if ((r = set_smem_attr(topm_fn(p, m), topm_smem(p, m)))) return r;
  if ((r = run_prep(p, X, log_weights, means, vars, o, ws, s))) return r;
  double* ll_dev = o.loglik_on_host ? reinterpret_cast<double*>(ws + p.off_ll) : total_loglik;
  if ((r = run_topm(p, X, m, resp_out, idx_out, ll_dev, ws, ts, s, log_weights, means, vars, o.topm_refine)))
    return r;
  if (o.loglik_on_host) {
    CUDA_TRY(cudaMemcpyAsync(total_loglik, ll_dev, sizeof(double), cudaMemcpyDeviceToHost, s));
    return sync_status(ws, s);
  }
  return GMM_OK;
}

int gmm_assign_threshold(const void* X, int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype,
                         const float* log_weights, const float* means, const float* vars, float tau,
                         int32_t max_per_point, int64_t* offsets, int32_t* idx_out, float* resp_out,
                         int64_t capacity, const gmm_opts* opts, void* stream) {
  g_launches = 0;
  gmm_opts o;
  gmm_default_opts(&o);
  if (opts) o = *opts;
  if (!X) return fail(GMM_ERR_INVALID_ARG, "X is NULL");
  int r;
  if ((r = check_ptr(log_weights, "log_weights")) || (r = check_ptr(means, "means")) ||
      (r = check_ptr(vars, "vars")))
    return r;
  if (!offsets || (reinterpret_cast<uintptr_t>(offsets) & 7))
    return fail(GMM_ERR_INVALID_ARG, "offsets must be a non-NULL 8-byte aligned device pointer");
  if (capacity < 0) return fail(GMM_ERR_INVALID_ARG, "capacity must be >= 0");
  if (capacity > 0 && ((r = check_ptr(idx_out, "idx_out")) || (r = check_ptr(resp_out, "resp_out")))) return r;
  if (!(tau > 0.f && tau <= 1.f)) return fail(GMM_ERR_INVALID_ARG, "tau must be in (0, 1]");
  if (max_per_point < 1 || max_per_point > 16) return fail(GMM_ERR_UNSUPPORTED, "max_per_point must be in [1, 16]");
  if (max_per_point > K) return fail(GMM_ERR_INVALID_ARG, "max_per_point must not exceed K");
  Plan p;
  if ((r = make_plan(p, X, N, D, K, cov_type, x_dtype, o, true))) return r;
  const int m = max_per_point;
  const int64_t n_blocks = (N + kThreshBlock - 1) / kThreshBlock;
  if (n_blocks > 0x7fffffffLL) return fail(GMM_ERR_UNSUPPORTED, "N too large for gmm_assign_threshold (grid limit)");
  // workspace: the EM workspace, the top-m lists of every point, block totals
  const size_t off_r = p.ws_bytes;
  const size_t off_i = off_r + align256(sizeof(float) * static_cast<size_t>(N) * m);
  const size_t off_b = off_i + align256(sizeof(int32_t) * static_cast<size_t>(N) * m);
  TopmSpace ts = topm_space(p, m, off_b + align256(sizeof(int64_t) * static_cast<size_t>(n_blocks + 1)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = nullptr;
  if ((r = get_workspace(ts.end, &ws))) return r;
  if ((r = set_smem_attr(topm_fn(p, m), topm_smem(p, m)))) return r;
  if ((r = run_prep(p, X, log_weights, means, vars, o, ws, s))) return r;
  float* tr = reinterpret_cast<float*>(ws + off_r);
  int32_t* ti = reinterpret_cast<int32_t*>(ws + off_i);
  int64_t* bt = reinterpret_cast<int64_t*>(ws + off_b);
  if ((r = run_topm(p, X, m, tr, ti, nullptr, ws, ts, s, log_weights, means, vars, o.topm_refine))) return r;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  if ((r = launch(kernel_handle(K_THRESH_COUNT), dim3(static_cast<unsigned>(n_blocks)), dim3(kThreshBlock), 0, s, 1,
                  static_cast<const float*>(tr), N, m, tau, offsets, bt)))
    return r;
  if ((r = launch(kernel_handle(K_THRESH_SCAN), dim3(1), dim3(1024), 0, s, 1, bt, n_blocks))) return r;
  if ((r = launch(kernel_handle(K_THRESH_SCATTER), dim3(static_cast<unsigned>(n_blocks)), dim3(kThreshBlock), 0, s,
                  1, static_cast<const float*>(tr), static_cast<const int32_t*>(ti), N, m, tau, offsets,
                  static_cast<const int64_t*>(bt), n_blocks, idx_out, resp_out, capacity, status)))
    return r;
  if (o.loglik_on_host) return sync_status(ws, s);
  return GMM_OK;
}

int gmm_stream_status(void* stream) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  uint8_t* buf = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    auto it = g_ws.find(dev);
    if (it == g_ws.end() || !it->second.buf) return GMM_OK;
    buf = it->second.buf;
  }
  uint32_t st[2] = {0, 0};
  CUDA_TRY(cudaMemcpy(st, buf, sizeof(st), cudaMemcpyDeviceToHost));
  if (st[0]) CUDA_TRY(cudaMemset(buf, 0, sizeof(st)));
  return status_to_code(st[0], st[1]);
}

void gmm_profile_begin(void) {
  for (auto& e : g_prof_events) {
    cudaEventDestroy(e.first);
    cudaEventDestroy(e.second);
  }
  g_prof_events.clear();
  g_prof_launches = 0;
  g_prof_on = true;
}

int gmm_profile_end(double* main_kernel_ms, int32_t* launches) {
  g_prof_on = false;
  double tot = 0.0;
  int rc = GMM_OK;
  for (auto& e : g_prof_events) {
    float ms = 0.f;
    if (rc == GMM_OK) {
      cudaError_t err = cudaEventSynchronize(e.second);
      if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e.first, e.second);
      if (err != cudaSuccess) rc = fail(GMM_ERR_CUDA, std::string("profile events: ") + cudaGetErrorString(err));
    }
    tot += ms;
    cudaEventDestroy(e.first);
    cudaEventDestroy(e.second);
  }
  g_prof_events.clear();
  if (main_kernel_ms) *main_kernel_ms = tot;
  if (launches) *launches = g_prof_launches;
  g_prof_launches = 0;
  return rc;
}

void gmm_release(void) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  for (auto& kv : g_ws) {
    if (kv.second.buf) {
      int cur = 0;
      cudaGetDevice(&cur);
      cudaSetDevice(kv.first);
      cudaDeviceSynchronize();
      cudaFree(kv.second.buf);
      cudaSetDevice(cur);
    }
  }
  g_ws.clear();
  std::lock_guard<std::mutex> lk2(g_pipe_mu);
  for (auto& kv : g_pipes) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(kv.first);
    HostPipe& hp = kv.second;
    cudaStreamSynchronize(hp.copy);
    for (int b = 0; b < 2; ++b) {
      cudaEventDestroy(hp.copied[b]);
      cudaEventDestroy(hp.freed[b]);
    }
    cudaEventDestroy(hp.start);
    cudaStreamDestroy(hp.copy);
    cudaSetDevice(cur);
  }
  g_pipes.clear();
}

}  // extern "C"

// ====================================================================== no-allocation variant
// gmm_em_step_noalloc: the single-pass EM step with all of its scratch taken
// from one fixed device array that is part of this library's module, for
// callers that must not call cudaMalloc/cudaFree while they run.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library reserves kNoAllocScratchBytes for it until the process exits.  Host
// code cannot use the variable's name as a device address; its address on
// each device is looked up once with cudaGetSymbolAddress (on the first call
// made with that device current) and cached.
constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;   // 24 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
uint8_t* g_noalloc_base[kNoAllocMaxDevices] = {};
std::mutex g_noalloc_mu;

// Address of the scratch array on the current device (looked up once).
int noalloc_scratch(uint8_t** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(GMM_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_base[dev]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr)
      return fail(GMM_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    g_noalloc_base[dev] = static_cast<uint8_t*>(ptr);
  }
  *out = g_noalloc_base[dev];
  return GMM_OK;
}

// Scratch layout of gmm_em_step_noalloc inside the fixed array; the number of
// tile groups (and so of CTAs) is lowered until the per-group statistics fit.
int noalloc_layout(Plan& p) {
  const size_t piece = static_cast<size_t>(2 * p.nch) * kChunkBytes;
  const size_t row_bytes = sizeof(double) * static_cast<size_t>(p.K_pad) * p.F;
  size_t fixed = kStatusBytes + align256(sizeof(Meta)) + 256 +
                 align256(static_cast<size_t>(p.n_slices) * p.np * piece) +
                 align256(static_cast<size_t>(p.n_slices) * kConstBytes) + 2 * align256(sizeof(float) * p.K_pad) +
                 align256(sizeof(double) * kCombineBlocks);
  if (fixed + align256(row_bytes) > kNoAllocScratchBytes)
    return fail(GMM_ERR_UNSUPPORTED, "problem too large for the 24 MiB scratch of gmm_em_step_noalloc");
  const int tg_fit = static_cast<int>((kNoAllocScratchBytes - fixed) / row_bytes);
  p.tg = std::max(1, std::min(p.tg, tg_fit));
  size_t off = kStatusBytes;
  p.off_meta = off; off += align256(sizeof(Meta));
  p.off_ll = off; off += 256;
  p.off_pimg = off; off += align256(static_cast<size_t>(p.n_slices) * p.np * piece);
  p.off_cimg = off; off += align256(static_cast<size_t>(p.n_slices) * kConstBytes);
  p.off_cadj = off; off += align256(sizeof(float) * p.K_pad);
  p.off_iscale = off; off += align256(sizeof(float) * p.K_pad);
  p.off_llpart = off; off += align256(sizeof(double) * std::max<size_t>(static_cast<size_t>(p.tg) * p.C, kCombineBlocks));
  p.off_part = off; off += align256(row_bytes * p.tg);
  p.off_lsepart = p.off_lse = off;
  if (off > kNoAllocScratchBytes) return fail(GMM_ERR_UNSUPPORTED, "scratch layout overflow");

  return GMM_OK;
}
}  // namespace

extern "C" int gmm_em_step_noalloc(const void* X, int64_t N, int32_t D, int32_t K, int32_t cov_type,
                                   int32_t x_dtype, const float* log_weights, const float* means,
                                   const float* vars, float* new_log_weights, float* new_means,
                                   float* new_vars, double* total_loglik, const gmm_opts* opts,
                                   void* stream) {
  g_launches = 0;
  gmm_opts o;
  gmm_default_opts(&o);
  if (opts) o = *opts;
  if (!X) return fail(GMM_ERR_INVALID_ARG, "X is NULL");
  int r;
  if ((r = check_ptr(log_weights, "log_weights")) || (r = check_ptr(means, "means")) ||
      (r = check_ptr(vars, "vars")) || (r = check_ptr(new_log_weights, "new_log_weights")) ||
      (r = check_ptr(new_means, "new_means")) || (r = check_ptr(new_vars, "new_vars")))
    return r;
  if (!total_loglik) return fail(GMM_ERR_INVALID_ARG, "total_loglik is NULL");
  if (cov_type == GMM_TIED) return fail(GMM_ERR_UNSUPPORTED, "gmm_em_step_noalloc supports spherical and diagonal covariance");
  o.plan = GMM_PLAN_CLUSTER;   // the single pass: no N-sized buffer
  Plan p;
  if (o.approx_top_k != 0 && o.approx_top_k < K)
    return fail(GMM_ERR_UNSUPPORTED, "gmm_em_step_noalloc runs exact EM only (approx_top_k must be 0 or >= K)");
  if ((r = make_plan(p, X, N, D, K, cov_type, x_dtype, o, true))) return r;
  if (p.two_pass)
    return fail(GMM_ERR_UNSUPPORTED, "gmm_em_step_noalloc supports K <= 1024 (larger K needs an N-sized buffer)");

  if ((r = noalloc_layout(p))) return r;
  uint8_t* ws = nullptr;
  if ((r = noalloc_scratch(&ws))) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* fn = estep_fn(p, MODE_EM);
  if ((r = set_smem_attr(fn, p.smem))) return r;
  // the array keeps the previous call's contents: clear the status words and
  // the statistics accumulators, which must start at zero
  CUDA_TRY(cudaMemsetAsync(ws, 0, 2 * sizeof(uint32_t), s));
  if ((r = run_prep(p, X, log_weights, means, vars, o, ws, s))) return r;
  const size_t row_bytes = sizeof(double) * static_cast<size_t>(p.K_pad) * p.F;
  CUDA_TRY(cudaMemsetAsync(ws + p.off_part, 0, row_bytes * p.tg, s));
  FusedArgs a = base_args(p, X, ws);
  a.mode = MODE_EM;
  a.C = p.C;
  if ((r = launch(fn, dim3(p.C * p.tg, 1), dim3(p.threads), p.smem, s, p.C, a))) return r;
  double* ll_dev = o.loglik_on_host ? reinterpret_cast<double*>(ws + p.off_ll) : total_loglik;
  {
    float reg = o.reg_covar, floor_ = o.var_floor;
    int Dp = p.nch * kAtomElems;
    if ((r = launch(kernel_handle(K_FINALIZE), dim3(p.K), dim3(128), 0, s, 1,
                    static_cast<const double*>(a.part), p.tg, p.K_pad, p.F, Dp, p.D, p.K, p.N, p.cov_diag, reg,
                    floor_, static_cast<double>(p.fast ? kRScale<1>() : kRScale<2>()), static_cast<const Meta*>(a.meta),
                    reinterpret_cast<const double*>(ws + p.off_llpart), p.tg * p.C, new_log_weights, new_means,
                    new_vars, means, vars, ll_dev, static_cast<double*>(nullptr))))
      return r;
  }
  if (o.loglik_on_host) {
    CUDA_TRY(cudaMemcpyAsync(total_loglik, ll_dev, sizeof(double), cudaMemcpyDeviceToHost, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    uint32_t st[2] = {0, 0};
    CUDA_TRY(cudaMemcpy(st, ws, sizeof(st), cudaMemcpyDeviceToHost));
    if (st[0]) return status_to_code(st[0], st[1]);
  }
  return GMM_OK;
}

extern "C" int gmm_plan_info(int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype,
                             const gmm_opts* opts, int32_t* info) {
  if (!info) return fail(GMM_ERR_INVALID_ARG, "info is NULL");
  gmm_opts o;
  gmm_default_opts(&o);
  if (opts) o = *opts;
  Plan p;
  int r;
  if ((r = make_plan(p, nullptr, N, D, K, cov_type, x_dtype, o, true))) return r;
  info[0] = p.two_pass ? p.C1e : p.C;
  info[1] = p.tg;
  info[2] = p.two_pass ? 1 : 0;
  info[3] = p.two_pass ? p.tg1e : 0;
  info[4] = p.flush;
  info[5] = p.threads;
  info[6] = 0;
  info[7] = p.n_tiles;
  if (cov_type != GMM_TIED) {
    gmm_opts on = o;
    on.plan = GMM_PLAN_CLUSTER;
    Plan pn;
    if (make_plan(pn, nullptr, N, D, K, cov_type, x_dtype, on, true) == GMM_OK && !pn.two_pass &&
        noalloc_layout(pn) == GMM_OK)
      info[6] = pn.tg;
  }
  return GMM_OK;
}
