// verkv_noalloc.cu -- verkv_certify_noalloc: the sketch logits and the certificate/selection
// kernels of verkv_attend_verified, for callers that cannot allocate device memory.
//
// The logits that the score kernel writes and the certify kernel reads are the only scratch these
// two kernels need.  Here they live in one fixed array in the library's own device memory instead
// of a caller workspace, so a call needs no context and no allocation.  The kernels are the same
// ones verkv_attend_verified launches, with the same launch shapes.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "verkv_internal.h"

using namespace verkv;

// The scratch: logits [units * q_per_kv][n].  Every call overwrites every logit it later reads,
// so nothing in it has to start at zero.  Every call on a GPU shares it.
static __device__ __align__(256) float g_logits[VERKV_NOALLOC_MAX_LOGITS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_logits_dev[kMaxDevices] = {};  // device address of g_logits, per device

// Set-up, once per device, with that device current: host code sees g_logits only as a host-side
// stand-in, so the kernels get the address the runtime reports for the device copy.
cudaError_t logits_address(int device, float **out) {
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_logits_dev[device]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_logits);
        if (e != cudaSuccess) return e;
        g_logits_dev[device] = static_cast<float *>(p);
    }
    *out = g_logits_dev[device];
    return cudaSuccess;
}

// Puts the caller's current device back when the call returns, on every path.
class DeviceRestore {
  public:
    DeviceRestore() { ok_ = cudaGetDevice(&saved_) == cudaSuccess; }
    ~DeviceRestore() {
        if (ok_) cudaSetDevice(saved_);
    }
    bool ok() const { return ok_; }

  private:
    int saved_ = 0;
    bool ok_ = false;
};

}  // namespace

extern "C" verkv_status verkv_certify_noalloc(int device, void *stream, int32_t units,
                                              int32_t q_per_kv, int32_t head_dim, int32_t n,
                                              const void *q, const void *sketch,
                                              const float *r_full, float eps, float delta,
                                              verkv_head_stats *stats_out, uint32_t *F_out,
                                              uint32_t *err_out) {
    const int G = q_per_kv;
    if (units < 1 || !(G == 1 || G == 2 || G == 4 || G == 8) ||
        !(head_dim == 64 || head_dim == 128) || n < 1 || n > 131072)
        return VERKV_EINVAL;
    if (!q || !sketch || !r_full || !stats_out || !F_out || !err_out) return VERKV_EINVAL;
    // q is read in 16-byte vectors and the sketch by bulk copies: both need 16-byte alignment;
    // the rest are read and written as 4-byte words.
    if ((((uintptr_t)q | (uintptr_t)sketch) & 15u) ||
        (((uintptr_t)r_full | (uintptr_t)stats_out | (uintptr_t)F_out | (uintptr_t)err_out) & 3u))
        return VERKV_EINVAL;
    if (!(eps > 0.0f) || !isfinite(eps) || !(delta > 0.0f) || !(delta < 1.0f)) return VERKV_EINVAL;
    if ((int64_t)units * G * n > (int64_t)VERKV_NOALLOC_MAX_LOGITS) return VERKV_ETOOLARGE;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return VERKV_ECUDA;
    if (device < 0 || device >= ndev || device >= kMaxDevices) return VERKV_EINVAL;
    DeviceRestore restore;
    if (!restore.ok()) return VERKV_ECUDA;
    if (cudaSetDevice(device) != cudaSuccess) return VERKV_ECUDA;
    float *logits = nullptr;
    if (logits_address(device, &logits) != cudaSuccess) return VERKV_ECUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(err_out, 0, sizeof(uint32_t), s) != cudaSuccess) return VERKV_ECUDA;

    // One "layer" of `units` consecutive units: unit_global(u) = u, query head qh = u * G + g.
    LayerIdx li{};
    li.layers = 1;
    li.layer = 0;
    li.kv_heads = units;
    li.G = G;

    ScoreArgs sa{};
    sa.sketch = static_cast<const uint16_t *>(sketch);
    sa.q = static_cast<const uint16_t *>(q);
    sa.scores = logits;
    sa.err = err_out;
    sa.n = n;
    sa.d = head_dim;
    sa.scale = (float)(1.0 / sqrt((double)head_dim));
    sa.li = li;
    if (launch_score(sa, units, s, false) != cudaSuccess) return VERKV_ECUDA;

    CertifyArgs ca{};
    ca.sel_gather = 1;
    ca.scores = logits;
    ca.r_full = r_full;
    ca.resident = nullptr;  // not read by the certify kernel
    ca.F = F_out;
    ca.qstats = stats_out;
    ca.err = err_out;
    ca.n = n;
    ca.W = (n + 31) / 32;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return VERKV_ECUDA;
    ca.cl = certify_cluster_size(n, units * G, sms);
    ca.chunk = certify_chunk(n, ca.cl);
    ca.eps = eps;
    ca.ldelta = (float)log(2.0 / (double)delta);
    ca.li = li;
    if (launch_certify(ca, units * G, certify_smem_bytes(ca.chunk), s) != cudaSuccess)
        return VERKV_ECUDA;
    return VERKV_OK;
}
