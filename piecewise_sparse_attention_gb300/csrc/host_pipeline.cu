// pisa_attention_host: the whole block-wise path (statistics, route, forward)
// on Q, K, V held in host memory, with the output written back to host
// memory, as one C call.
//
// Heads are independent, so they go through in contiguous groups. An upload
// stream copies group c + 1 to the device while a compute stream runs the
// three calls on group c and a download stream copies group c - 1's output
// back; two compute streams alternate so that one group's last CTAs overlap
// the next group's first. Device buffers (inputs, statistics, route, output)
// are two groups deep and come from the caller's workspace; the streams and
// events are created for the call and released when their work is done.
#include <math.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pisa.h"
#include "common.cuh"

namespace {

constexpr int kMaxGroups = 64;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t dt_size(int dt) { return dt == PISA_BF16 ? 2 : 4; }

// Bounds of `groups` contiguous head groups; with `taper` the first and the
// last group weigh half as much as the others (their copies are the ones the
// pipeline cannot hide). Returns the number of groups.
int head_group_bounds(int heads, int groups, int taper, int* bounds) {
  const int g = groups < 1 ? 1 : (groups > heads ? heads : groups);
  double wts[kMaxGroups];
  for (int i = 0; i < g; ++i) wts[i] = 1.0;
  if (taper && g >= 3) wts[0] = wts[g - 1] = 0.5;
  double tot = 0.0;
  for (int i = 0; i < g; ++i) tot += wts[i];
  double acc = 0.0;
  bounds[0] = 0;
  for (int i = 1; i < g; ++i) {
    acc += wts[i - 1];
    int b = static_cast<int>(nearbyint(acc * heads / tot));
    if (b < bounds[i - 1] + 1) b = bounds[i - 1] + 1;
    if (b > heads - (g - i)) b = heads - (g - i);
    bounds[i] = b;
  }
  bounds[g] = heads;
  return g;
}

struct Layout {
  size_t q, k, v, o, qbar, kbar, idx, cnt;  // byte offsets of buffer 0
  size_t per_buffer;                        // bytes of one buffer set
};

Layout layout(int in_dtype, int out_dtype, int width, int n, int d, int max_sel) {
  const size_t nb = static_cast<size_t>(pisa::ceil_div(n, pisa::kBlock));
  const size_t in_bytes = align256(static_cast<size_t>(width) * n * d * dt_size(in_dtype));
  Layout L;
  L.q = 0;
  L.k = L.q + in_bytes;
  L.v = L.k + in_bytes;
  L.o = L.v + in_bytes;
  L.qbar = L.o + align256(static_cast<size_t>(width) * n * d * dt_size(out_dtype));
  L.kbar = L.qbar + align256(static_cast<size_t>(width) * nb * d * 4);
  L.idx = L.kbar + align256(static_cast<size_t>(width) * nb * d * 4);
  L.cnt = L.idx + align256(static_cast<size_t>(width) * nb * max_sel * 4);
  L.per_buffer = L.cnt + align256(static_cast<size_t>(width) * nb * 4);
  return L;
}

int max_sel_of(int n, int topk, int band) {
  const long long nb = pisa::ceil_div(n, pisa::kBlock);
  const long long need = static_cast<long long>(topk) + 2LL * band + 1LL;
  return static_cast<int>(need < nb ? need : nb);
}

// Streams and events of one call, destroyed at scope exit (the runtime frees
// them once their enqueued work has completed).
struct Resources {
  cudaStream_t up = nullptr, down = nullptr, comp[2] = {nullptr, nullptr};
  cudaEvent_t ev[8] = {};
  ~Resources() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);
    for (cudaStream_t s : {up, down, comp[0], comp[1]})
      if (s) cudaStreamDestroy(s);
  }
};

}  // namespace

extern "C" {

size_t pisa_attention_host_workspace_size(int in_dtype, int out_dtype, int heads, int n, int d,
                                          int topk, int band, int groups, int taper) {
  if (heads < 1 || n < 1 || topk < 0 || band < 0) return 0;
  int bounds[kMaxGroups + 1];
  const int g = head_group_bounds(heads, groups < kMaxGroups ? groups : kMaxGroups, taper, bounds);
  int width = 0;
  for (int c = 0; c < g; ++c) width = bounds[c + 1] - bounds[c] > width ? bounds[c + 1] - bounds[c] : width;
  return 2 * layout(in_dtype, out_dtype, width, n, d, max_sel_of(n, topk, band)).per_buffer;
}

int pisa_attention_host(const void* q, const void* k, const void* v, int in_dtype, int heads,
                        int n, int d, int block, float scale, int topk, int band, void* out,
                        int out_dtype, int groups, int taper, void* workspace,
                        size_t workspace_bytes, int32_t* dev_status, void* stream) {
  nvtxRangePushA("pisa_attention_host");
  struct Pop {
    ~Pop() { nvtxRangePop(); }
  } pop;
  if (!q || !k || !v || !out) return PISA_ERR_INVALID_ARG;
  if ((in_dtype != PISA_F32 && in_dtype != PISA_BF16) ||
      (out_dtype != PISA_F32 && out_dtype != PISA_BF16))
    return PISA_ERR_INVALID_ARG;
  if (heads < 1 || n < 1 || block != pisa::kBlock || topk < 0 || band < 0 || groups < 1 ||
      groups > kMaxGroups || !(scale > 0.f) || !isfinite(scale))
    return PISA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PISA_ERR_UNSUPPORTED;
  int bounds[kMaxGroups + 1];
  const int g = head_group_bounds(heads, groups, taper, bounds);
  int width = 0;
  for (int c = 0; c < g; ++c) width = bounds[c + 1] - bounds[c] > width ? bounds[c + 1] - bounds[c] : width;
  const int max_sel = max_sel_of(n, topk, band);
  const Layout L = layout(in_dtype, out_dtype, width, n, d, max_sel);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < 2 * L.per_buffer) {
    pisa::note_error("pisa_attention_host: needs a 256-byte aligned workspace of %zu bytes",
                     2 * L.per_buffer);
    return PISA_ERR_INVALID_ARG;
  }
  const int nb = pisa::ceil_div(n, pisa::kBlock);
  const size_t in_head = static_cast<size_t>(n) * d * dt_size(in_dtype);
  const size_t out_head = static_cast<size_t>(n) * d * dt_size(out_dtype);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  auto buf = [&](int b, size_t off) { return ws + b * L.per_buffer + off; };
  cudaStream_t caller = static_cast<cudaStream_t>(stream);

  Resources R;
  for (cudaStream_t* s : {&R.up, &R.down, &R.comp[0], &R.comp[1]})
    PISA_CUDA_TRY(cudaStreamCreateWithFlags(s, cudaStreamNonBlocking));
  for (cudaEvent_t& e : R.ev) PISA_CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  cudaEvent_t start = R.ev[0], loaded = R.ev[1];
  cudaEvent_t consumed[2] = {R.ev[2], R.ev[3]};  // compute done with buffer b
  cudaEvent_t drained[2] = {R.ev[4], R.ev[5]};   // output of buffer b copied back
  bool used[2] = {false, false};

  // everything already on the caller's stream comes first
  PISA_CUDA_TRY(cudaEventRecord(start, caller));
  for (cudaStream_t s : {R.up, R.down, R.comp[0], R.comp[1]})
    PISA_CUDA_TRY(cudaStreamWaitEvent(s, start, 0));

  for (int c = 0; c < g; ++c) {
    const int h0 = bounds[c], w = bounds[c + 1] - bounds[c], b = c % 2;
    // upload group c into buffer b once the compute of group c - 2 has read it
    if (used[b]) PISA_CUDA_TRY(cudaStreamWaitEvent(R.up, consumed[b], 0));
    const void* src[3] = {q, k, v};
    const size_t off[3] = {L.q, L.k, L.v};
    for (int t = 0; t < 3; ++t)
      PISA_CUDA_TRY(cudaMemcpyAsync(buf(b, off[t]),
                                    static_cast<const unsigned char*>(src[t]) + h0 * in_head,
                                    w * in_head, cudaMemcpyHostToDevice, R.up));
    PISA_CUDA_TRY(cudaEventRecord(loaded, R.up));
    // stats, route and forward of group c on its compute stream
    cudaStream_t cs = R.comp[b];
    PISA_CUDA_TRY(cudaStreamWaitEvent(cs, loaded, 0));
    if (used[b]) PISA_CUDA_TRY(cudaStreamWaitEvent(cs, drained[b], 0));
    float* qbar = reinterpret_cast<float*>(buf(b, L.qbar));
    float* kbar = reinterpret_cast<float*>(buf(b, L.kbar));
    int32_t* idx = reinterpret_cast<int32_t*>(buf(b, L.idx));
    int32_t* cnt = reinterpret_cast<int32_t*>(buf(b, L.cnt));
    int rc = pisa_block_stats(buf(b, L.q), buf(b, L.k), buf(b, L.v), in_dtype, w, n, d, block,
                              qbar, kbar, nullptr, nullptr, PISA_F32, dev_status, cs);
    if (rc == PISA_OK)
      rc = pisa_route(qbar, kbar, w, nb, d, scale, topk, band, idx, cnt, max_sel, dev_status, cs);
    if (rc == PISA_OK)
      rc = pisa_forward(buf(b, L.q), buf(b, L.k), buf(b, L.v), in_dtype, w, n, d, block, scale,
                        idx, cnt, max_sel, buf(b, L.o), out_dtype, dev_status, cs);
    if (rc != PISA_OK) return rc;
    PISA_CUDA_TRY(cudaEventRecord(consumed[b], cs));
    // download group c's output
    PISA_CUDA_TRY(cudaStreamWaitEvent(R.down, consumed[b], 0));
    PISA_CUDA_TRY(cudaMemcpyAsync(static_cast<unsigned char*>(out) + h0 * out_head, buf(b, L.o),
                                  w * out_head, cudaMemcpyDeviceToHost, R.down));
    PISA_CUDA_TRY(cudaEventRecord(drained[b], R.down));
    used[b] = true;
  }
  // the caller's stream continues after every stream of the call
  const cudaStream_t all[4] = {R.up, R.down, R.comp[0], R.comp[1]};
  const cudaEvent_t fin[4] = {R.ev[6], R.ev[7], consumed[0], consumed[1]};
  for (int s = 0; s < 4; ++s) {
    PISA_CUDA_TRY(cudaEventRecord(fin[s], all[s]));
    PISA_CUDA_TRY(cudaStreamWaitEvent(caller, fin[s], 0));
  }
  return PISA_OK;
}

}  // extern "C"
