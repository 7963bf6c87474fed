// C ABI entry points: argument validation (synchronous, nothing enqueued on error) and
// dispatch to the launchers. No exception crosses this boundary.
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "ns_small.h"

namespace mao {

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
int g_cc[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

void query_device(int dev) {
  std::call_once(g_dev_once[dev], [dev] {
    int sms = 0, major = 0, minor = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    g_sms[dev] = sms > 0 ? sms : 1;
    g_cc[dev] = major * 10 + minor;
  });
}

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}
}  // namespace

int num_sms() {
  const int d = current_device();
  query_device(d);
  return g_sms[d];
}

int device_cc() {
  const int d = current_device();
  query_device(d);
  return g_cc[d];
}

namespace {
std::atomic<long long> g_launches{0};

struct Profile {
  bool on = false;
  int32_t cap = 0;
  int32_t used = 0;
  std::vector<cudaEvent_t> ev;  // 2 per launch
  std::vector<int32_t> tag;     // 1 per launch
};
Profile g_prof;
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
std::atomic<unsigned long long> g_wait_limit{4000000000ull};  // 4 s
}  // namespace

unsigned long long wait_limit_ns() { return g_wait_limit.load(std::memory_order_relaxed); }

void profile_before_launch(cudaStream_t stream, int tag) {
  if (g_prof.on && g_prof.used < g_prof.cap) {
    g_prof.tag[g_prof.used] = tag;
    cudaEventRecord(g_prof.ev[2 * g_prof.used], stream);
  }
}

void profile_after_launch(cudaStream_t stream) {
  if (g_prof.on && g_prof.used < g_prof.cap) {
    cudaEventRecord(g_prof.ev[2 * g_prof.used + 1], stream);
    ++g_prof.used;
  }
}

namespace {
Profile g_span;  // event pairs around whole runs of tensor-core products
}  // namespace

void profile_span_begin(cudaStream_t stream) {
  if (g_span.on && g_span.used < g_span.cap) cudaEventRecord(g_span.ev[2 * g_span.used], stream);
}

void profile_span_end(cudaStream_t stream) {
  if (g_span.on && g_span.used < g_span.cap) {
    cudaEventRecord(g_span.ev[2 * g_span.used + 1], stream);
    ++g_span.used;
  }
}

}  // namespace mao

using namespace mao;

extern "C" {

int32_t mao_abi_version(void) { return 1; }

const char* mao_status_string(mao_status s) {
  switch (s) {
    case MAO_OK: return "MAO_OK";
    case MAO_ERR_INVALID_ARG: return "MAO_ERR_INVALID_ARG";
    case MAO_ERR_UNSUPPORTED: return "MAO_ERR_UNSUPPORTED";
    case MAO_ERR_MISALIGNED: return "MAO_ERR_MISALIGNED";
    case MAO_ERR_WORKSPACE: return "MAO_ERR_WORKSPACE";
    case MAO_ERR_CUDA: return "MAO_ERR_CUDA";
    case MAO_ERR_TIMEOUT: return "MAO_ERR_TIMEOUT";
    case MAO_ERR_NUMERIC: return "MAO_ERR_NUMERIC";
  }
  return "MAO_ERR_UNKNOWN";
}

mao_status muon_momentum_update(const mao_mat* M, const mao_mat* G, int32_t batch, float mu,
                                void* stream) {
  if (!M || !G || batch < 1 || !std::isfinite(mu)) return MAO_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    mao_status st = check_mat(M[b]);
    if (st == MAO_OK) st = check_mat(G[b]);
    if (st != MAO_OK) return st;
    if (M[b].rows != G[b].rows || M[b].cols != G[b].cols) return MAO_ERR_INVALID_ARG;
  }
  return momentum_launch(M, G, batch, mu, static_cast<cudaStream_t>(stream));
}

size_t ns_workspace_bytes(const mao_mat* X, int32_t batch, int32_t compute) {
  if (!X || batch < 1 || !valid_dtype(compute)) return 0;
  for (int b = 0; b < batch; ++b) {
    if (X[b].rows < 1 || X[b].cols < 1 || X[b].rows > (int64_t(1) << 31) ||
        X[b].cols > (int64_t(1) << 31))
      return 0;
  }
  return ns_workspace_size(X, batch, compute);
}

mao_status ns_orthogonalize(const mao_mat* in, const mao_mat* out, int32_t batch, int32_t steps,
                            const float* coeffs, int32_t coeff_stride, float eps,
                            int32_t compute, uint32_t* const* sign_bits, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!in || !out || batch < 1 || steps < 1 || steps > 64 || !coeffs) return MAO_ERR_INVALID_ARG;
  if (coeff_stride != 0 && coeff_stride != 3) return MAO_ERR_INVALID_ARG;
  if (!valid_dtype(compute) || !std::isfinite(eps) || eps < 0.0f) return MAO_ERR_INVALID_ARG;
  for (int i = 0; i < (coeff_stride ? 3 * steps : 3); ++i)
    if (!std::isfinite(coeffs[i])) return MAO_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    mao_status st = check_ns_input(in[b]);
    if (st != MAO_OK) return st;
    const bool bits = sign_bits && sign_bits[b];
    st = check_mat(out[b], bits);
    if (st != MAO_OK) return st;
    if (out[b].rows != in[b].rows || out[b].cols != in[b].cols) return MAO_ERR_INVALID_ARG;
    if (bits && (reinterpret_cast<uintptr_t>(sign_bits[b]) % 4 != 0)) return MAO_ERR_MISALIGNED;
  }
  if (!workspace) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MAO_ERR_MISALIGNED;
  if (compute == MAO_BF16 && device_cc() / 10 != 10) return MAO_ERR_UNSUPPORTED;
  if (workspace_bytes < ns_workspace_size(in, batch, compute)) return MAO_ERR_WORKSPACE;
  return ns_run(in, out, batch, steps, coeffs, coeff_stride, eps, compute, sign_bits, workspace,
                workspace_bytes, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
// Argument checks of muon_step (and muon_step_host): MAO_OK when the step may be enqueued.
mao_status muon_step_check(const mao_mat* W, const mao_mat* M, const mao_mat* G,
                           const mao_mat* W_out, int32_t batch, float mu, float lr,
                           int32_t steps, const float* coeffs, int32_t coeff_stride, float eps,
                           int32_t compute, const void* workspace, size_t workspace_bytes) {
  if (!W || !M || !G || batch < 1 || steps < 1 || steps > 64 || !coeffs) return MAO_ERR_INVALID_ARG;
  if (coeff_stride != 0 && coeff_stride != 3) return MAO_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.0f || !std::isfinite(mu) || !std::isfinite(lr))
    return MAO_ERR_INVALID_ARG;
  for (int i = 0; i < (coeff_stride ? 3 * steps : 3); ++i)
    if (!std::isfinite(coeffs[i])) return MAO_ERR_INVALID_ARG;
  if (compute != MAO_BF16) return MAO_ERR_UNSUPPORTED;
  for (int b = 0; b < batch; ++b) {
    mao_status st = check_mat(W[b]);
    if (st == MAO_OK) st = check_mat(M[b]);
    if (st == MAO_OK) st = check_mat(G[b]);
    if (st != MAO_OK) return st;
    if (M[b].rows != W[b].rows || M[b].cols != W[b].cols || G[b].rows != W[b].rows ||
        G[b].cols != W[b].cols)
      return MAO_ERR_INVALID_ARG;
    if (W_out) {
      st = check_mat(W_out[b]);
      if (st != MAO_OK) return st;
      if (W_out[b].rows != W[b].rows || W_out[b].cols != W[b].cols ||
          W_out[b].dtype != W[b].dtype)
        return MAO_ERR_INVALID_ARG;
    }
  }
  if (!workspace) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MAO_ERR_MISALIGNED;
  if (device_cc() / 10 != 10) return MAO_ERR_UNSUPPORTED;
  if (workspace_bytes < ns_workspace_size(M, batch, compute)) return MAO_ERR_WORKSPACE;
  return MAO_OK;
}
}  // namespace

extern "C" {

mao_status muon_step(const mao_mat* W, const mao_mat* M, const mao_mat* G, const mao_mat* W_out,
                     int32_t batch, float mu, float lr, int32_t steps, const float* coeffs,
                     int32_t coeff_stride, float eps, int32_t compute, void* workspace,
                     size_t workspace_bytes, void* stream) {
  const mao_status st = muon_step_check(W, M, G, W_out, batch, mu, lr, steps, coeffs,
                                        coeff_stride, eps, compute, workspace, workspace_bytes);
  if (st != MAO_OK) return st;
  const NsFuse fuse{G, W_out ? W : nullptr, mu, lr};
  return ns_run(M, W_out ? W_out : W, batch, steps, coeffs, coeff_stride, eps, compute, nullptr,
                workspace, workspace_bytes, static_cast<cudaStream_t>(stream), &fuse);
}

mao_status muon_step_host(const mao_mat* W, const mao_mat* M, const mao_mat* G,
                          const mao_mat* W_out, int32_t batch, float mu, float lr, int32_t steps,
                          const float* coeffs, int32_t coeff_stride, float eps, int32_t compute,
                          void* workspace, size_t workspace_bytes, const void* g_host,
                          void* g_dev, size_t g_bytes, void* w_host, const void* w_dev,
                          size_t w_bytes, void* stream, void* wait_event, void* record_event) {
  if ((g_bytes && (!g_host || !g_dev)) || (w_bytes && (!w_host || !w_dev)))
    return MAO_ERR_INVALID_ARG;
  mao_status st = muon_step_check(W, M, G, W_out, batch, mu, lr, steps, coeffs, coeff_stride,
                                  eps, compute, workspace, workspace_bytes);
  if (st != MAO_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (g_bytes && cudaMemcpyAsync(g_dev, g_host, g_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MAO_ERR_CUDA;
  if (wait_event &&
      cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(wait_event), 0) != cudaSuccess)
    return MAO_ERR_CUDA;
  const NsFuse fuse{G, W_out ? W : nullptr, mu, lr};
  st = ns_run(M, W_out ? W_out : W, batch, steps, coeffs, coeff_stride, eps, compute, nullptr,
              workspace, workspace_bytes, s, &fuse);
  if (st != MAO_OK) return st;
  if (record_event && cudaEventRecord(static_cast<cudaEvent_t>(record_event), s) != cudaSuccess)
    return MAO_ERR_CUDA;
  if (w_bytes && cudaMemcpyAsync(w_host, w_dev, w_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MAO_ERR_CUDA;
  return MAO_OK;
}

mao_status sign_muon_step(const mao_mat* W, const mao_mat* M, const mao_mat* G,
                          int32_t n_workers, uint32_t* words, int64_t worker_stride_words,
                          uint32_t* vote, float mu, float lr, int32_t steps, const float* coeffs,
                          int32_t coeff_stride, float eps, int32_t compute, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!W || !M || !G || !words || !vote || n_workers < 1 || n_workers > 65535 || steps < 1 ||
      steps > 64 || !coeffs)
    return MAO_ERR_INVALID_ARG;
  if (coeff_stride != 0 && coeff_stride != 3) return MAO_ERR_INVALID_ARG;
  if (!valid_dtype(compute) || !std::isfinite(eps) || eps < 0.0f || !std::isfinite(mu) ||
      !std::isfinite(lr))
    return MAO_ERR_INVALID_ARG;
  for (int i = 0; i < (coeff_stride ? 3 * steps : 3); ++i)
    if (!std::isfinite(coeffs[i])) return MAO_ERR_INVALID_ARG;
  mao_status st = check_mat(*W);
  if (st != MAO_OK) return st;
  const int64_t nbits = W->rows * W->cols;
  if (worker_stride_words < ceil_div(nbits, 32)) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(words) % 4 != 0 || reinterpret_cast<uintptr_t>(vote) % 4 != 0)
    return MAO_ERR_MISALIGNED;
  std::vector<mao_mat> out(n_workers);
  std::vector<uint32_t*> bits(n_workers);
  for (int m = 0; m < n_workers; ++m) {
    st = check_mat(M[m]);
    if (st == MAO_OK) st = check_mat(G[m]);
    if (st != MAO_OK) return st;
    if (M[m].rows != W->rows || M[m].cols != W->cols || G[m].rows != W->rows ||
        G[m].cols != W->cols)
      return MAO_ERR_INVALID_ARG;
    out[m] = M[m];
    out[m].data = nullptr;  // signs only
    bits[m] = words + int64_t(m) * worker_stride_words;
  }
  if (!workspace) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MAO_ERR_MISALIGNED;
  if (compute == MAO_BF16 && device_cc() / 10 != 10) return MAO_ERR_UNSUPPORTED;
  if (workspace_bytes < ns_workspace_size(M, n_workers, compute)) return MAO_ERR_WORKSPACE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // small fp32 matrices: the momentum inside the one-launch Newton–Schulz kernel; on the
  // tensor-core path inside the pass that stages M for the products; otherwise its own
  // launch first. Then the vote and the update of W in one launch.
  if (ns_small_eligible(M, out.data(), n_workers, steps, compute)) {
    st = ns_small_run(M, out.data(), n_workers, steps, coeffs, coeff_stride, eps, bits.data(), s,
                      G, mu);
  } else if (compute == MAO_BF16) {
    NsFuse fuse{G, nullptr, mu, 0.0f};
    fuse.update = false;
    st = ns_run(M, out.data(), n_workers, steps, coeffs, coeff_stride, eps, compute, bits.data(),
                workspace, workspace_bytes, s, &fuse);
  } else {
    st = momentum_launch(M, G, n_workers, mu, s);
    if (st == MAO_OK)
      st = ns_run(M, out.data(), n_workers, steps, coeffs, coeff_stride, eps, compute,
                  bits.data(), workspace, workspace_bytes, s);
  }
  if (st == MAO_OK)
    st = vote_update_launch(words, n_workers, worker_stride_words, nbits, vote, *W, lr, s);
  return st;
}

mao_status sign_pack_bits(const mao_mat* U, uint32_t* bits, void* stream) {
  if (!U || !bits) return MAO_ERR_INVALID_ARG;
  const mao_status st = check_mat(*U);
  if (st != MAO_OK) return st;
  if (reinterpret_cast<uintptr_t>(bits) % 4 != 0) return MAO_ERR_MISALIGNED;
  return sign_pack_launch(*U, bits, static_cast<cudaStream_t>(stream));
}

mao_status majority_vote_packed(const uint32_t* bits, int32_t n_workers,
                                int64_t worker_stride_words, int64_t nbits, uint32_t* vote,
                                void* stream) {
  if (!bits || !vote || n_workers < 1 || n_workers > 65535 || nbits < 1) return MAO_ERR_INVALID_ARG;
  if (worker_stride_words < ceil_div(nbits, 32)) return MAO_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(bits) % 4 != 0 || reinterpret_cast<uintptr_t>(vote) % 4 != 0)
    return MAO_ERR_MISALIGNED;
  return vote_launch(bits, n_workers, worker_stride_words, nbits, vote,
                     static_cast<cudaStream_t>(stream));
}

mao_status sign_int8(const mao_mat* U, int8_t* s, void* stream) {
  if (!U || !s) return MAO_ERR_INVALID_ARG;
  const mao_status st = check_mat(*U);
  if (st != MAO_OK) return st;
  return sign_int8_launch(*U, s, static_cast<cudaStream_t>(stream));
}

mao_status majority_vote_int8(const int8_t* s, int32_t n_workers, int64_t worker_stride,
                              int64_t n, int8_t* sum, int8_t* s_bar, uint32_t* vote,
                              void* stream) {
  if (!s || n_workers < 1 || n_workers > 127 || n < 1 || worker_stride < n) return MAO_ERR_INVALID_ARG;
  if (!sum && !s_bar && !vote) return MAO_ERR_INVALID_ARG;
  if (vote && reinterpret_cast<uintptr_t>(vote) % 4 != 0) return MAO_ERR_MISALIGNED;
  return vote_int8_launch(s, n_workers, worker_stride, n, sum, s_bar, vote,
                          static_cast<cudaStream_t>(stream));
}

mao_status apply_update(const mao_mat* W, const uint32_t* const* vote, const mao_mat* U,
                        int32_t batch, float lr, void* stream) {
  if (!W || batch < 1 || !std::isfinite(lr)) return MAO_ERR_INVALID_ARG;
  if ((vote == nullptr) == (U == nullptr)) return MAO_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    mao_status st = check_mat(W[b]);
    if (st != MAO_OK) return st;
    if (vote) {
      if (!vote[b]) return MAO_ERR_INVALID_ARG;
      if (reinterpret_cast<uintptr_t>(vote[b]) % 4 != 0) return MAO_ERR_MISALIGNED;
    } else {
      st = check_mat(U[b]);
      if (st != MAO_OK) return st;
      if (U[b].rows != W[b].rows || U[b].cols != W[b].cols) return MAO_ERR_INVALID_ARG;
    }
  }
  return update_launch(W, vote, U, batch, lr, static_cast<cudaStream_t>(stream));
}

void mao_set_wait_limit(uint64_t ns) { g_wait_limit.store(ns, std::memory_order_relaxed); }

uint64_t mao_get_wait_limit(void) { return g_wait_limit.load(std::memory_order_relaxed); }

mao_status mao_sync_status(void* stream) {
  const mao_status a = tc_read_and_clear_error(static_cast<cudaStream_t>(stream));
  const mao_status b = dion_read_and_clear_error(static_cast<cudaStream_t>(stream));
  const mao_status c = small_read_and_clear_error(static_cast<cudaStream_t>(stream));
  if (a == MAO_ERR_CUDA || b == MAO_ERR_CUDA || c == MAO_ERR_CUDA) return MAO_ERR_CUDA;
  return a != MAO_OK ? a : b != MAO_OK ? b : c;
}

int64_t mao_launch_count(void) { return g_launches.load(); }

mao_status mao_profile_begin(int32_t max_launches) {
  if (max_launches < 1 || max_launches > (1 << 20) || g_prof.on) return MAO_ERR_INVALID_ARG;
  g_prof.ev.assign(size_t(2) * max_launches, nullptr);
  for (auto& e : g_prof.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      for (auto& x : g_prof.ev)
        if (x) cudaEventDestroy(x);
      g_prof.ev.clear();
      return MAO_ERR_CUDA;
    }
  }
  g_prof.tag.assign(size_t(max_launches), 0);
  g_prof.cap = max_launches;
  g_prof.used = 0;
  g_prof.on = true;
  return MAO_OK;
}

mao_status mao_profile_span_begin(int32_t max_spans) {
  if (max_spans < 1 || max_spans > (1 << 20) || g_span.on) return MAO_ERR_INVALID_ARG;
  g_span.ev.assign(size_t(2) * max_spans, nullptr);
  for (auto& e : g_span.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      for (auto& f : g_span.ev)
        if (f) cudaEventDestroy(f);
      g_span.ev.clear();
      return MAO_ERR_CUDA;
    }
  }
  g_span.cap = max_spans;
  g_span.used = 0;
  g_span.on = true;
  return MAO_OK;
}

int32_t mao_profile_span_end(float* ms_out, int32_t max_out) {
  if (!g_span.on) return 0;
  g_span.on = false;
  const int32_t n = g_span.used;
  bool ok = true;
  for (int32_t i = 0; i < n; ++i) {
    float ms = 0.0f;
    if (cudaEventSynchronize(g_span.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_span.ev[2 * i], g_span.ev[2 * i + 1]) != cudaSuccess)
      ok = false;
    if (ms_out && i < max_out) ms_out[i] = ms;
  }
  for (auto& e : g_span.ev) cudaEventDestroy(e);
  g_span.ev.clear();
  g_span.used = 0;
  return ok ? n : -1;
}

int32_t mao_profile_end(float* ms_out, int32_t max_out) {
  return mao_profile_end_tagged(ms_out, nullptr, max_out);
}

int32_t mao_profile_end_tagged(float* ms_out, int32_t* tags_out, int32_t max_out) {
  if (!g_prof.on) return 0;
  g_prof.on = false;
  int32_t n = g_prof.used;
  bool ok = true;
  for (int32_t i = 0; i < n; ++i) {
    float ms = 0.0f;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess)
      ok = false;
    if (ms_out && i < max_out) ms_out[i] = ms;
    if (tags_out && i < max_out) tags_out[i] = g_prof.tag[i];
  }
  for (auto& e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.clear();
  g_prof.used = 0;
  return ok ? n : -1;
}

}  // extern "C"
