// libbeamboundary: C ABI of the fused sublayer boundary (see include/beam_boundary.h).
//
// Host side: argument validation (before any CUDA call), the launch shape
// (vectors per thread, CTA size, persistent grid from the occupancy of the
// chosen kernel on this device), the residual coefficients c1 = RN32(sqrt((n-1)/n))
// and c2 = RN32(1/sqrt(n)) evaluated in double, the error factor that lets the
// kernel certify the rounding of its compensated row sums, and the launch.
#include "beam_boundary.h"

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "boundary_kernels.cuh"

namespace {

using beam::BoundaryParams;
using KernelFn = void (*)(BoundaryParams);

constexpr int kMaxDevices = 64;
constexpr int kMaxVpt = 8;

__device__ unsigned int g_status_word;  // device-side error word (bounded waits)

struct DeviceInfo {
    bool checked = false;
    bool ok = false;
    int sms = 0;
    int occ[2][kMaxVpt + 1][beam::kMaxThreads / 32 + 1] = {};  // resident CTAs per SM, 0 = unknown
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

template <bool MOE>
KernelFn kernel_for(int vpt) {
    switch (vpt) {
    case 1: return beam::boundary_kernel<1, MOE>;
    case 2: return beam::boundary_kernel<2, MOE>;
    case 3: return beam::boundary_kernel<3, MOE>;
    case 4: return beam::boundary_kernel<4, MOE>;
    case 5: return beam::boundary_kernel<5, MOE>;
    case 6: return beam::boundary_kernel<6, MOE>;
    case 7: return beam::boundary_kernel<7, MOE>;
    case 8: return beam::boundary_kernel<8, MOE>;
    default: return nullptr;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

int round_up32(int v) { return (v + 31) & ~31; }

// CTA size for `vpt` vectors per thread, or 0 when the row does not fit
int threads_for(int nvec, int vpt) {
    int nt = round_up32((nvec + vpt - 1) / vpt);
    return nt <= beam::kMaxThreads ? nt : 0;
}

// Automatic vectors per thread: the first candidate whose CTA wastes under
// 1/16 of its slots, else the smallest that fits.
int choose_vpt(int nvec, bool moe) {
    static const int dense_pref[] = {4, 2, 5, 3, 6, 8, 1, 7};
    static const int moe_pref[] = {2, 1, 3, 4, 5, 6, 8, 7};
    const int* pref = moe ? moe_pref : dense_pref;
    for (int i = 0; i < 8; ++i) {
        int v = pref[i], nt = threads_for(nvec, v);
        if (nt && (nt * v - nvec) * 16 <= nvec) return v;
    }
    for (int v = 1; v <= kMaxVpt; ++v)
        if (threads_for(nvec, v)) return v;
    return 0;
}

// Bound on |c - c_exact| / (u^2 T) for the compensated sum, u = 2^-24, T the
// exact sum. Terms are >= 0. A lane adds m terms with TwoSum and a rounded
// compensation: error <= 0.505 m (m+1) u^2 T, |c| <= 1.01 m u T. Every merge
// level (lane pair, 5 shuffle levels, nw-1 sequential block merges) adds
// <= 2 (g + 1.01) u^2 T and raises the |c| bound g by 1.01 u T. The factor
// 1.5 is slack; 1 + 2^-10 covers T <= s (1 + 2^-10).
float error_factor(int vpt, int nt) {
    const double u = std::ldexp(1.0, -24);
    double m = 4.0 * vpt;
    double g = 1.01 * m, E = 0.505 * m * (m + 1.0);
    int levels = 1 + 5 + (nt / 32 - 1);
    for (int i = 0; i < levels; ++i) {
        g += 1.01;
        E += 2.0 * g;
    }
    return (float)(E * u * u * 1.5 * (1.0 + 1.0 / 1024.0));
}

beam_status current_device(int* dev_out, DeviceInfo** info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return BEAM_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.checked) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return BEAM_ERR_CUDA;
        }
        d.ok = (major == 10 && minor == 3);
        d.sms = sms;
        d.checked = true;
    }
    if (!d.ok) return BEAM_ERR_DEVICE;
    *dev_out = dev;
    *info = &d;
    return BEAM_OK;
}

beam_status resident_ctas(DeviceInfo* d, bool moe, int vpt, int nt, KernelFn fn, int* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    int& slot = d->occ[moe ? 1 : 0][vpt][nt / 32];
    if (slot == 0) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, reinterpret_cast<const void*>(fn), nt, 0) !=
            cudaSuccess) {
            cudaGetLastError();
            return BEAM_ERR_CUDA;
        }
        slot = nb > 0 ? nb : 1;
    }
    *out = slot;
    return BEAM_OK;
}

beam_status check_common(int n, float eps, int64_t T, int D, const beam_launch_opts* opts) {
    if (T < 0 || D < 8 || (D & 7) || D > BEAM_MAX_D || T > (int64_t(1) << 40)) return BEAM_ERR_SHAPE;
    if (n < 1 || !(eps >= 0.0f) || !std::isfinite(eps)) return BEAM_ERR_ARG;
    if (opts) {
        if (opts->vec_per_thread < 0 || opts->vec_per_thread > kMaxVpt || opts->ctas_per_sm < 0 ||
            (opts->flags & ~BEAM_OPT_FORCE_EXACT_SUM))
            return BEAM_ERR_ARG;
        if (opts->vec_per_thread && !threads_for(D / 8, opts->vec_per_thread)) return BEAM_ERR_ARG;
    }
    return BEAM_OK;
}

beam_status launch(bool moe, beam_stream_t stream, uint16_t* h, const uint16_t* x, const uint16_t* e,
                   const float* w, const uint16_t* post_w, const uint16_t* pre_w, int n, float eps,
                   int64_t T, int D, uint16_t* y, const beam_launch_opts* opts) {
    int dev = 0;
    DeviceInfo* info = nullptr;
    beam_status st = current_device(&dev, &info);
    if (st != BEAM_OK) return st;

    const int nvec = D / 8;
    const int vpt = (opts && opts->vec_per_thread) ? opts->vec_per_thread : choose_vpt(nvec, moe);
    const int nt = threads_for(nvec, vpt);
    KernelFn fn = moe ? kernel_for<true>(vpt) : kernel_for<false>(vpt);
    if (!fn || !nt) return BEAM_ERR_SHAPE;

    int per_sm = 0;
    st = resident_ctas(info, moe, vpt, nt, fn, &per_sm);
    if (st != BEAM_OK) return st;
    if (opts && opts->ctas_per_sm) per_sm = opts->ctas_per_sm < per_sm ? opts->ctas_per_sm : per_sm;
    int64_t grid = (int64_t)per_sm * info->sms;
    if (grid > T) grid = T;

    BoundaryParams p;
    p.h = h;
    p.x = x;
    p.e = e;
    p.w = w;
    p.post_w = post_w;
    p.pre_w = pre_w;
    p.y = y;
    p.T = T;
    p.D = D;
    p.nvec = nvec;
    p.c1 = (float)std::sqrt((double)(n - 1) / (double)n);
    p.c2 = (float)(1.0 / std::sqrt((double)n));
    p.eps = eps;
    p.errk = error_factor(vpt, nt);
    p.flags = (opts && (opts->flags & BEAM_OPT_FORCE_EXACT_SUM)) ? beam::kFlagForceExact : 0u;

    void* args[] = {&p};
    cudaError_t err = cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3((unsigned)grid), dim3(nt), args,
                                       0, reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    return BEAM_OK;
}

}  // namespace

extern "C" {

beam_status beam_boundary_fused_ex(beam_stream_t stream, uint16_t* h, const uint16_t* x,
                                   const uint16_t* post_w, const uint16_t* pre_w, int n, float eps,
                                   int64_t T, int D, uint16_t* y_out, const beam_launch_opts* opts) {
    beam_status st = check_common(n, eps, T, D, opts);
    if (st != BEAM_OK || T == 0) return st;
    if (!h || !x || !post_w || !pre_w || !y_out) return BEAM_ERR_NULL;
    if (!aligned16(h) || !aligned16(x) || !aligned16(post_w) || !aligned16(pre_w) || !aligned16(y_out))
        return BEAM_ERR_ALIGN;
    const size_t rows = (size_t)T * (size_t)D * 2u, vec = (size_t)D * 2u;
    if (overlaps(y_out, rows, h, rows) || overlaps(y_out, rows, x, rows) || overlaps(y_out, rows, post_w, vec) ||
        overlaps(y_out, rows, pre_w, vec))
        return BEAM_ERR_ALIAS;
    if ((const void*)x != (const void*)h && overlaps(h, rows, x, rows)) return BEAM_ERR_ALIAS;
    if (overlaps(h, rows, post_w, vec) || overlaps(h, rows, pre_w, vec)) return BEAM_ERR_ALIAS;
    return launch(false, stream, h, x, nullptr, nullptr, post_w, pre_w, n, eps, T, D, y_out, opts);
}

beam_status beam_boundary_fused(beam_stream_t stream, uint16_t* h, const uint16_t* x, const uint16_t* post_w,
                                const uint16_t* pre_w, int n, float eps, int64_t T, int D, uint16_t* y_out) {
    return beam_boundary_fused_ex(stream, h, x, post_w, pre_w, n, eps, T, D, y_out, nullptr);
}

beam_status beam_moe_combine_boundary_ex(beam_stream_t stream, uint16_t* h, const uint16_t* expert_out,
                                         const float* topk_w, const uint16_t* post_w, const uint16_t* pre_w,
                                         int n, float eps, int64_t T, int D, uint16_t* y_out,
                                         const beam_launch_opts* opts) {
    beam_status st = check_common(n, eps, T, D, opts);
    if (st != BEAM_OK || T == 0) return st;
    if (!h || !expert_out || !topk_w || !post_w || !pre_w || !y_out) return BEAM_ERR_NULL;
    if (!aligned16(h) || !aligned16(expert_out) || !aligned16(topk_w) || !aligned16(post_w) ||
        !aligned16(pre_w) || !aligned16(y_out))
        return BEAM_ERR_ALIGN;
    const size_t rows = (size_t)T * (size_t)D * 2u, vec = (size_t)D * 2u;
    const size_t erows = rows * BEAM_MOE_TOPK, wbytes = (size_t)T * BEAM_MOE_TOPK * 4u;
    if (overlaps(y_out, rows, h, rows) || overlaps(y_out, rows, expert_out, erows) ||
        overlaps(y_out, rows, topk_w, wbytes) || overlaps(y_out, rows, post_w, vec) ||
        overlaps(y_out, rows, pre_w, vec))
        return BEAM_ERR_ALIAS;
    if (overlaps(h, rows, expert_out, erows) || overlaps(h, rows, topk_w, wbytes) || overlaps(h, rows, post_w, vec) ||
        overlaps(h, rows, pre_w, vec))
        return BEAM_ERR_ALIAS;
    return launch(true, stream, h, nullptr, expert_out, topk_w, post_w, pre_w, n, eps, T, D, y_out, opts);
}

beam_status beam_moe_combine_boundary(beam_stream_t stream, uint16_t* h, const uint16_t* expert_out,
                                      const float* topk_w, const uint16_t* post_w, const uint16_t* pre_w, int n,
                                      float eps, int64_t T, int D, uint16_t* y_out) {
    return beam_moe_combine_boundary_ex(stream, h, expert_out, topk_w, post_w, pre_w, n, eps, T, D, y_out,
                                        nullptr);
}

beam_status beam_sync_status(beam_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    unsigned int word = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_status_word, sizeof word, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    return word ? BEAM_ERR_TIMEOUT : BEAM_OK;
}

beam_status beam_exact_sum_count(beam_stream_t stream, uint64_t* count, int reset) {
    if (!count) return BEAM_ERR_NULL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long v = 0, zero = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&v, beam::g_exact_sum_count, sizeof v, 0, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        (reset && cudaMemcpyToSymbolAsync(beam::g_exact_sum_count, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                          s) != cudaSuccess) ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    *count = v;
    return BEAM_OK;
}

const char* beam_status_string(beam_status status) {
    switch (status) {
    case BEAM_OK: return "ok";
    case BEAM_ERR_NULL: return "a required pointer is NULL";
    case BEAM_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case BEAM_ERR_SHAPE: return "bad shape: need T >= 0 and D a multiple of 8 in [8, BEAM_MAX_D]";
    case BEAM_ERR_ARG: return "bad argument: need n >= 1, finite eps >= 0 and valid options";
    case BEAM_ERR_ALIAS: return "output overlaps an input, or h partly overlaps an input";
    case BEAM_ERR_CUDA: return "a CUDA runtime call failed";
    case BEAM_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case BEAM_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    }
    return "unknown status";
}

int beam_version(void) { return 10000; }

}  // extern "C"
