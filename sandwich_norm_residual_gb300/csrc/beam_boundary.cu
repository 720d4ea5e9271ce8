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
#include <initializer_list>
#include <mutex>
#include <utility>

#include "boundary_kernels.cuh"
#include "route.cuh"
#include "qk_norm.cuh"

namespace {

using beam::BoundaryParams;
using KernelFn = void (*)(BoundaryParams);

constexpr int kMaxDevices = 64;
constexpr int kMaxVpt = 8;
constexpr int kMaxPrefetch = 8;
constexpr int kAutoPrefetch = 1;       // rows ahead prefetched into L2 (register kernels)
constexpr int kAutoStages = -1;        // dense: registers + L2 prefetch measured faster than the ring
constexpr int kTestStages = 2;         // ring slots when only the wait test hook asks for the ring
constexpr uint64_t kWaitNs = 2000000000ull;    // every mbarrier wait gives up after 2 s
constexpr uint64_t kTestWaitNs = 1000000ull;   // the test hook's wait: 1 ms

enum KernelKind { kDenseRegs = 0, kMoeRegs = 1, kDenseRing = 2 };

struct OccKey {
    KernelFn fn;
    int nt, smem;
};

struct DeviceInfo {
    bool checked = false;
    bool ok = false;
    int ordinal = 0;
    bool pageable_access = false;             // kernels may read pageable host memory
    int sms = 0;
    long long l2_bytes = 0;
    int smem_optin = 0;                       // max dynamic + static shared memory per CTA
    KernelFn lim_fn[64] = {};                 // kernels whose dynamic smem limit was raised
    int lim_val[64] = {};
    int lim_n = 0;
    OccKey occ_key[128] = {};
    int occ_val[128] = {};
    int occ_n = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// FULL kernels (row = exactly NT * VPT vectors, weights staged in shared
// memory) exist for these vectors-per-thread values
bool has_full(int vpt) { return vpt >= 2 && vpt <= 5; }

template <int V, int KIND, bool FULL, bool QUANT>
KernelFn pick() {
    if constexpr (KIND == kDenseRing) return beam::boundary_ring_kernel<V, FULL>;
    else return beam::boundary_kernel<V, KIND == kMoeRegs, FULL, QUANT>;
}

template <int KIND, bool QUANT>
KernelFn kernel_for(int vpt, bool full) {
    if (full) {
        switch (vpt) {
        case 2: return pick<2, KIND, true, QUANT>();
        case 3: return pick<3, KIND, true, QUANT>();
        case 4: return pick<4, KIND, true, QUANT>();
        case 5: return pick<5, KIND, true, QUANT>();
        default: return nullptr;
        }
    }
    switch (vpt) {
    case 1: return pick<1, KIND, false, QUANT>();
    case 2: return pick<2, KIND, false, QUANT>();
    case 3: return pick<3, KIND, false, QUANT>();
    case 4: return pick<4, KIND, false, QUANT>();
    case 5: return pick<5, KIND, false, QUANT>();
    case 6: return pick<6, KIND, false, QUANT>();
    case 7: return pick<7, KIND, false, QUANT>();
    case 8: return pick<8, KIND, false, QUANT>();
    default: return nullptr;
    }
}

KernelFn kernel_for_kind(int kind, int vpt, bool full, bool quant = false) {
    if (quant) return kind == kMoeRegs ? kernel_for<kMoeRegs, true>(vpt, full) : kernel_for<kDenseRegs, true>(vpt, full);
    return kind == kDenseRing ? kernel_for<kDenseRing, false>(vpt, full)
           : kind == kMoeRegs ? kernel_for<kMoeRegs, false>(vpt, full)
                              : kernel_for<kDenseRegs, false>(vpt, full);
}

// NVFP4 destination of y (NULL: y is written as BF16)
struct QuantOut {
    uint8_t* q;
    uint8_t* sf;
    float gs;
};

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

// Automatic vectors per thread: the first preferred value whose CTA wastes
// under 1/16 of its slots, else the smallest that fits. The preferences come
// from sweeps at D = 5120 on GB300 (dense: 5 -> 128 threads; MoE: 2 -> 320).
int choose_vpt(int nvec, bool moe) {
    static const int dense_pref[] = {5, 4, 6, 3, 2, 8, 7, 1};
    static const int moe_pref[] = {2, 3, 4, 1, 5, 6, 8, 7};
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
float error_factor_terms(double m, int levels) {
    const double u = std::ldexp(1.0, -24);
    double g = 1.01 * m, E = 0.505 * m * (m + 1.0);
    for (int i = 0; i < levels; ++i) {
        g += 1.01;
        E += 2.0 * g;
    }
    return (float)(E * u * u * 1.5 * (1.0 + 1.0 / 1024.0));
}

float error_factor(int vpt, int nt) { return error_factor_terms(4.0 * vpt, 1 + 5 + (nt / 32 - 1)); }

beam_status current_device(DeviceInfo** info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return BEAM_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.checked) {
        int major = 0, minor = 0, sms = 0, optin = 0, pageable = 0, l2 = 0;
        if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            cudaGetLastError();
            return BEAM_ERR_CUDA;
        }
        d.ok = (major == 10 && minor == 3);
        d.ordinal = dev;
        d.l2_bytes = l2;
        d.pageable_access = pageable != 0;
        d.sms = sms;
        d.smem_optin = optin;
        d.checked = true;
    }
    if (!d.ok) return BEAM_ERR_DEVICE;
    *info = &d;
    return BEAM_OK;
}

// Dynamic shared memory `fn` may use (the opt-in maximum less its static
// shared memory); raises the kernel's limit to it on first use.
beam_status smem_limit(DeviceInfo* d, KernelFn fn, int* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < d->lim_n; ++i)
        if (d->lim_fn[i] == fn) {
            *out = d->lim_val[i];
            return BEAM_OK;
        }
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, reinterpret_cast<const void*>(fn)) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    int limit = d->smem_optin - (int)attr.sharedSizeBytes;
    if (limit < 0) limit = 0;
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             limit) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    if (d->lim_n < 64) {
        d->lim_fn[d->lim_n] = fn;
        d->lim_val[d->lim_n++] = limit;
    }
    *out = limit;
    return BEAM_OK;
}

// resident CTAs per SM of `fn` with `nt` threads and `smem` dynamic bytes (cached)
beam_status resident_ctas(DeviceInfo* d, KernelFn fn, int nt, int smem, int* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < d->occ_n; ++i) {
        const OccKey& k = d->occ_key[i];
        if (k.fn == fn && k.nt == nt && k.smem == smem) {
            *out = d->occ_val[i];
            return BEAM_OK;
        }
    }
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, reinterpret_cast<const void*>(fn), nt, smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    nb = nb > 0 ? nb : 1;
    if (d->occ_n < 128) {
        d->occ_key[d->occ_n] = OccKey{fn, nt, smem};
        d->occ_val[d->occ_n++] = nb;
    }
    *out = nb;
    return BEAM_OK;
}

beam_status check_common(int n, float eps, int64_t T, int D, const beam_launch_opts* opts) {
    if (T < 0 || D < 8 || (D & 7) || D > BEAM_MAX_D || T > (int64_t(1) << 40)) return BEAM_ERR_SHAPE;
    if (n < 1 || !(eps >= 0.0f) || !std::isfinite(eps)) return BEAM_ERR_ARG;
    if (opts) {
        if (opts->vec_per_thread < 0 || opts->vec_per_thread > kMaxVpt || opts->ctas_per_sm < 0 ||
            opts->prefetch_rows < -1 || opts->prefetch_rows > kMaxPrefetch || opts->stages < -1 ||
            opts->stages == 1 || opts->stages > beam::kMaxStages || opts->reserved[0] || opts->reserved[1] ||
            opts->reserved[2] || (opts->flags & ~(BEAM_OPT_FORCE_EXACT_SUM | BEAM_OPT_TEST_WAIT_TIMEOUT | BEAM_OPT_PDL)))
            return BEAM_ERR_ARG;
        if ((opts->flags & BEAM_OPT_TEST_WAIT_TIMEOUT) && opts->stages == -1) return BEAM_ERR_ARG;
        if (opts->vec_per_thread && !threads_for(D / 8, opts->vec_per_thread)) return BEAM_ERR_ARG;
    }
    return BEAM_OK;
}

beam_status launch(bool moe, beam_stream_t stream, uint16_t* h, const uint16_t* x, const uint16_t* e,
                   const float* w, const uint16_t* post_w, const uint16_t* pre_w, int n, float eps,
                   int64_t T, int D, uint16_t* y, const beam_launch_opts* opts, float route_scale = 1.0f,
                   const QuantOut* quant = nullptr) {
    DeviceInfo* info = nullptr;
    beam_status st = current_device(&info);
    if (st != BEAM_OK) return st;

    const int nvec = D / 8;
    const int vpt = (opts && opts->vec_per_thread) ? opts->vec_per_thread : choose_vpt(nvec, moe);
    const int nt = threads_for(nvec, vpt);
    if (!nt) return BEAM_ERR_SHAPE;

    // FULL: the row is exactly nt * vpt vectors; its kernels stage the norm
    // weights (4 D bytes, BF16) in shared memory
    const bool full = has_full(vpt) && nt * vpt == nvec;
    const int wbytes = full ? 4 * D : 0;
    const int slot_bytes = 4 * D;
    int kind = moe ? kMoeRegs : kDenseRing;
    int stages = 0;
    KernelFn fn = nullptr;
    int limit = 0;
    if (!moe) {
        // dense rows go through the shared-memory ring when at least two slots fit
        int want = (opts && opts->stages) ? opts->stages : kAutoStages;
        if (quant) want = -1;  // the NVFP4 output exists only in the register kernels
        if (want == -1 && opts && !opts->stages && (opts->flags & BEAM_OPT_TEST_WAIT_TIMEOUT)) want = kTestStages;
        if (want == -1) {
            kind = kDenseRegs;
        } else {
            fn = kernel_for_kind(kDenseRing, vpt, full);
            if (!fn) return BEAM_ERR_SHAPE;
            st = smem_limit(info, fn, &limit);
            if (st != BEAM_OK) return st;
            const int max_slots = (limit - wbytes) / slot_bytes;
            if (want <= max_slots) {
                stages = want;
            } else if (opts && opts->stages > 0) {
                return BEAM_ERR_ARG;  // asked for more slots than fit
            } else if (max_slots >= 2) {
                stages = max_slots < beam::kMaxStages ? max_slots : beam::kMaxStages;
            } else {
                if (opts && (opts->flags & BEAM_OPT_TEST_WAIT_TIMEOUT)) return BEAM_ERR_ARG;
                kind = kDenseRegs;
            }
        }
    }
    if (kind != kDenseRing) {
        fn = kernel_for_kind(kind, vpt, full, quant != nullptr);
        if (!fn) return BEAM_ERR_SHAPE;
        st = smem_limit(info, fn, &limit);
        if (st != BEAM_OK) return st;
        if (wbytes > limit) {  // weights do not fit: the generic kernel reads them from global memory
            fn = kernel_for_kind(kind, vpt, false, quant != nullptr);
            if (!fn) return BEAM_ERR_SHAPE;
        }
    }
    const bool full_used = (kind == kDenseRing) ? full : (full && wbytes <= limit);
    const int smem = (kind == kDenseRing ? stages * slot_bytes : 0) + (full_used ? wbytes : 0);

    const int prefetch = (opts && opts->prefetch_rows) ? (opts->prefetch_rows < 0 ? 0 : opts->prefetch_rows)
                                                       : kAutoPrefetch;
    int per_sm = 0;
    st = resident_ctas(info, fn, nt, smem, &per_sm);
    if (st != BEAM_OK) return st;
    if (opts && opts->ctas_per_sm) {
        per_sm = opts->ctas_per_sm < per_sm ? opts->ctas_per_sm : per_sm;
    } else if (kind != kDenseRing) {
        // rows in flight (each CTA's current row and its prefetched ones) stay
        // within half of L2; past that the prefetched rows are evicted before
        // use (measured on the MoE rows: 3 CTAs/SM re-read 4% and ran 11% slower)
        const long long row_in = moe ? (long long)D * 2 * (BEAM_MOE_TOPK + 1) + BEAM_MOE_TOPK * 4 : (long long)D * 4;
        const long long fit = (info->l2_bytes / 2) / ((long long)info->sms * (prefetch + 1) * row_in);
        if (fit < per_sm) per_sm = fit < 1 ? 1 : (int)fit;
    }
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
    p.flags = 0u;
    if (opts && (opts->flags & BEAM_OPT_FORCE_EXACT_SUM)) p.flags |= beam::kFlagForceExact;
    if (opts && (opts->flags & BEAM_OPT_TEST_WAIT_TIMEOUT)) p.flags |= beam::kFlagTestWaitTimeout;
    p.prefetch_rows = prefetch;
    p.stages = stages;
    p.wait_ns = kWaitNs;
    p.test_wait_ns = kTestWaitNs;
    p.route_scale = route_scale;
    p.yq = quant ? quant->q : nullptr;
    p.ysf = quant ? quant->sf : nullptr;
    p.y_gs = quant ? quant->gs : 0.0f;

    void* args[] = {&p};
    cudaError_t err;
    if (opts && (opts->flags & BEAM_OPT_PDL)) {
        // programmatic dependent launch: the kernel may start during the
        // previous kernel on the stream and waits for it after staging weights
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(nt);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = reinterpret_cast<cudaStream_t>(stream);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
    } else {
        err = cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3((unsigned)grid), dim3(nt), args,
                               (size_t)smem, reinterpret_cast<cudaStream_t>(stream));
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    return BEAM_OK;
}

// The address at which the current device's kernels reach `p`: device memory
// of this device and managed memory as is, page-locked host memory at its
// mapped device address, pageable host memory only where the device reads it
// through the host's page tables.
template <class P>
beam_status device_address(const DeviceInfo* info, P*& p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
        return a.device == info->ordinal ? BEAM_OK : BEAM_ERR_ARG;
    case cudaMemoryTypeManaged:
        return BEAM_OK;
    case cudaMemoryTypeHost:
        if (!a.devicePointer) return BEAM_ERR_ARG;
        p = static_cast<P*>(a.devicePointer);
        return BEAM_OK;
    default:
        return info->pageable_access ? BEAM_OK : BEAM_ERR_ARG;
    }
}

// Launch shape for operands in host memory: the register kernels, no L2
// prefetch (the rows stream over the CPU-GPU link).
const beam_launch_opts kHostOpts = {0u, 0, 0, -1, -1, {0, 0, 0}};

template <class... P>
beam_status host_addresses(P*&... ptrs) {
    DeviceInfo* info = nullptr;
    beam_status st = current_device(&info);
    if (st != BEAM_OK) return st;
    for (beam_status s : {device_address(info, ptrs)...})
        if (s != BEAM_OK) return s;
    return BEAM_OK;
}

}  // namespace

extern "C" {

static beam_status dense_boundary(beam_stream_t stream, uint16_t* h, const uint16_t* x, const uint16_t* post_w,
                                  const uint16_t* pre_w, int n, float eps, int64_t T, int D, uint16_t* y_out,
                                  const beam_launch_opts* opts, bool host) {
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
    if (host) {
        st = host_addresses(h, x, post_w, pre_w, y_out);
        if (st != BEAM_OK) return st;
        opts = &kHostOpts;
    }
    return launch(false, stream, h, x, nullptr, nullptr, post_w, pre_w, n, eps, T, D, y_out, opts);
}

beam_status beam_boundary_fused_ex(beam_stream_t stream, uint16_t* h, const uint16_t* x,
                                   const uint16_t* post_w, const uint16_t* pre_w, int n, float eps,
                                   int64_t T, int D, uint16_t* y_out, const beam_launch_opts* opts) {
    return dense_boundary(stream, h, x, post_w, pre_w, n, eps, T, D, y_out, opts, false);
}

beam_status beam_boundary_fused_host(beam_stream_t stream, uint16_t* h, const uint16_t* x, const uint16_t* post_w,
                                     const uint16_t* pre_w, int n, float eps, int64_t T, int D, uint16_t* y_out) {
    return dense_boundary(stream, h, x, post_w, pre_w, n, eps, T, D, y_out, nullptr, true);
}

static beam_status check_nvfp4(int64_t T, int D, float gs, const uint8_t* q, const uint8_t* sf,
                               const beam_launch_opts* opts) {
    if (D % 16) return BEAM_ERR_SHAPE;
    // the register kernels alone write NVFP4: no ring options
    if (opts && (opts->stages > 0 || (opts->flags & BEAM_OPT_TEST_WAIT_TIMEOUT))) return BEAM_ERR_ARG;
    if (!(gs > 0.0f) || !std::isfinite(gs)) return BEAM_ERR_ARG;
    if (T > 0 && (!q || !sf)) return BEAM_ERR_NULL;
    if (T > 0 && !aligned16(q)) return BEAM_ERR_ALIGN;
    if (overlaps(q, (size_t)T * D / 2, sf, (size_t)T * D / 16)) return BEAM_ERR_ALIAS;
    return BEAM_OK;
}

// y's NVFP4 buffers against every other operand
static bool nvfp4_overlaps(const uint8_t* q, const uint8_t* sf, int64_t T, int D,
                           std::initializer_list<std::pair<const void*, size_t>> others) {
    for (const auto& o : others)
        if (overlaps(q, (size_t)T * D / 2, o.first, o.second) || overlaps(sf, (size_t)T * D / 16, o.first, o.second))
            return true;
    return false;
}

beam_status beam_boundary_fused_nvfp4(beam_stream_t stream, uint16_t* h, const uint16_t* x, const uint16_t* post_w,
                                      const uint16_t* pre_w, int n, float eps, int64_t T, int D,
                                      float y_global_scale, uint8_t* y_fp4, uint8_t* y_scale,
                                      const beam_launch_opts* opts) {
    beam_status st = check_common(n, eps, T, D, opts);
    if (st == BEAM_OK) st = check_nvfp4(T, D, y_global_scale, y_fp4, y_scale, opts);
    if (st != BEAM_OK || T == 0) return st;
    if (!h || !x || !post_w || !pre_w) return BEAM_ERR_NULL;
    if (!aligned16(h) || !aligned16(x) || !aligned16(post_w) || !aligned16(pre_w)) return BEAM_ERR_ALIGN;
    const size_t rows = (size_t)T * (size_t)D * 2u, vec = (size_t)D * 2u;
    if (nvfp4_overlaps(y_fp4, y_scale, T, D, {{h, rows}, {x, rows}, {post_w, vec}, {pre_w, vec}}))
        return BEAM_ERR_ALIAS;
    if ((const void*)x != (const void*)h && overlaps(h, rows, x, rows)) return BEAM_ERR_ALIAS;
    if (overlaps(h, rows, post_w, vec) || overlaps(h, rows, pre_w, vec)) return BEAM_ERR_ALIAS;
    const QuantOut qo{y_fp4, y_scale, y_global_scale};
    return launch(false, stream, h, x, nullptr, nullptr, post_w, pre_w, n, eps, T, D, nullptr, opts, 1.0f, &qo);
}

beam_status beam_moe_combine_boundary_nvfp4(beam_stream_t stream, uint16_t* h, const uint16_t* expert_out,
                                            const float* topk_w, const uint16_t* post_w, const uint16_t* pre_w,
                                            int n, float eps, int64_t T, int D, float y_global_scale,
                                            uint8_t* y_fp4, uint8_t* y_scale, const beam_launch_opts* opts) {
    beam_status st = check_common(n, eps, T, D, opts);
    if (st == BEAM_OK) st = check_nvfp4(T, D, y_global_scale, y_fp4, y_scale, opts);
    if (st != BEAM_OK || T == 0) return st;
    if (!h || !expert_out || !topk_w || !post_w || !pre_w) return BEAM_ERR_NULL;
    if (!aligned16(h) || !aligned16(expert_out) || !aligned16(topk_w) || !aligned16(post_w) || !aligned16(pre_w))
        return BEAM_ERR_ALIGN;
    const size_t rows = (size_t)T * (size_t)D * 2u, vec = (size_t)D * 2u;
    const size_t erows = rows * BEAM_MOE_TOPK, wbytes = (size_t)T * BEAM_MOE_TOPK * 4u;
    if (nvfp4_overlaps(y_fp4, y_scale, T, D,
                       {{h, rows}, {expert_out, erows}, {topk_w, wbytes}, {post_w, vec}, {pre_w, vec}}))
        return BEAM_ERR_ALIAS;
    if (overlaps(h, rows, expert_out, erows) || overlaps(h, rows, topk_w, wbytes) || overlaps(h, rows, post_w, vec) ||
        overlaps(h, rows, pre_w, vec))
        return BEAM_ERR_ALIAS;
    const QuantOut qo{y_fp4, y_scale, y_global_scale};
    return launch(true, stream, h, nullptr, expert_out, topk_w, post_w, pre_w, n, eps, T, D, nullptr, opts, 1.0f,
                  &qo);
}

beam_status beam_boundary_fused(beam_stream_t stream, uint16_t* h, const uint16_t* x, const uint16_t* post_w,
                                const uint16_t* pre_w, int n, float eps, int64_t T, int D, uint16_t* y_out) {
    return beam_boundary_fused_ex(stream, h, x, post_w, pre_w, n, eps, T, D, y_out, nullptr);
}

static beam_status moe_boundary(beam_stream_t stream, uint16_t* h, const uint16_t* expert_out,
                                const float* topk_w, float route_scale, const uint16_t* post_w,
                                const uint16_t* pre_w, int n, float eps, int64_t T, int D, uint16_t* y_out,
                                const beam_launch_opts* opts, bool host = false) {
    beam_status st = check_common(n, eps, T, D, opts);
    if (st != BEAM_OK || T == 0) return st;
    if (!std::isfinite(route_scale)) return BEAM_ERR_ARG;
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
    if (host) {
        st = host_addresses(h, expert_out, topk_w, post_w, pre_w, y_out);
        if (st != BEAM_OK) return st;
        opts = &kHostOpts;
    }
    return launch(true, stream, h, nullptr, expert_out, topk_w, post_w, pre_w, n, eps, T, D, y_out, opts,
                  route_scale);
}

beam_status beam_moe_combine_boundary_host(beam_stream_t stream, uint16_t* h, const uint16_t* expert_out,
                                           const float* topk_w, const uint16_t* post_w, const uint16_t* pre_w,
                                           int n, float eps, int64_t T, int D, uint16_t* y_out) {
    return moe_boundary(stream, h, expert_out, topk_w, 1.0f, post_w, pre_w, n, eps, T, D, y_out, nullptr, true);
}

beam_status beam_moe_combine_boundary_ex(beam_stream_t stream, uint16_t* h, const uint16_t* expert_out,
                                         const float* topk_w, const uint16_t* post_w, const uint16_t* pre_w,
                                         int n, float eps, int64_t T, int D, uint16_t* y_out,
                                         const beam_launch_opts* opts) {
    return moe_boundary(stream, h, expert_out, topk_w, 1.0f, post_w, pre_w, n, eps, T, D, y_out, opts);
}

beam_status beam_moe_combine_boundary_scaled(beam_stream_t stream, uint16_t* h, const uint16_t* expert_out,
                                             const float* topk_w, float route_scale, const uint16_t* post_w,
                                             const uint16_t* pre_w, int n, float eps, int64_t T, int D,
                                             uint16_t* y_out) {
    return moe_boundary(stream, h, expert_out, topk_w, route_scale, post_w, pre_w, n, eps, T, D, y_out,
                        nullptr);
}

beam_status beam_moe_route_ex(beam_stream_t stream, const float* logits, const float* bias, int64_t T, int E,
                              int n_group, int topk_group, int topk, float route_scale, int32_t* topk_idx,
                              float* topk_w, uint32_t flags) {
    if (T < 0 || T > (int64_t(1) << 40) || E != BEAM_ROUTE_EXPERTS) return BEAM_ERR_SHAPE;
    if (n_group < 1 || n_group > 32 || (n_group & (n_group - 1)) || topk_group < 1 || topk_group > n_group ||
        topk < 1 || topk > BEAM_ROUTE_MAX_TOPK || topk > topk_group * (E / n_group) || !std::isfinite(route_scale) ||
        (flags & ~BEAM_OPT_PDL))
        return BEAM_ERR_ARG;
    if (T == 0) return BEAM_OK;
    if (!logits || !bias || !topk_idx || !topk_w) return BEAM_ERR_NULL;
    if (!aligned16(logits) || !aligned16(bias) || (reinterpret_cast<uintptr_t>(topk_idx) & 3u) ||
        (reinterpret_cast<uintptr_t>(topk_w) & 3u))
        return BEAM_ERR_ALIGN;
    const size_t zb = (size_t)T * (size_t)E * 4u, ob = (size_t)T * (size_t)topk * 4u, bb = (size_t)E * 4u;
    if (overlaps(topk_idx, ob, topk_w, ob) || overlaps(topk_idx, ob, logits, zb) || overlaps(topk_idx, ob, bias, bb) ||
        overlaps(topk_w, ob, logits, zb) || overlaps(topk_w, ob, bias, bb))
        return BEAM_ERR_ALIAS;
    DeviceInfo* info = nullptr;
    beam_status st = current_device(&info);
    if (st != BEAM_OK) return st;
    beam::RouteParams p;
    p.logits = logits;
    p.bias = bias;
    p.idx = topk_idx;
    p.w = topk_w;
    p.T = T;
    p.n_group = n_group;
    p.topk_group = topk_group;
    p.topk = topk;
    p.scale = route_scale;
    const int64_t blocks = (T + beam::kRouteWarps - 1) / beam::kRouteWarps;  // one token per warp
    if (blocks > 0x7FFFFFFF) return BEAM_ERR_SHAPE;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const void* fn = (n_group == 8 && topk_group == 4 && topk == 8)  // the Beam / DeepSeek-V3 router
                         ? reinterpret_cast<const void*>(beam::route_kernel<8, 4, 8>)
                         : reinterpret_cast<const void*>(beam::route_kernel<0, 0, 0>);
    void* args[] = {&p};
    cudaError_t err;
    if (flags & BEAM_OPT_PDL) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        cfg.stream = cs;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelExC(&cfg, fn, args);
    } else {
        err = cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(256), args, 0, cs);
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    return BEAM_OK;
}

beam_status beam_moe_route(beam_stream_t stream, const float* logits, const float* bias, int64_t T, int E,
                           int n_group, int topk_group, int topk, float route_scale, int32_t* topk_idx,
                           float* topk_w) {
    return beam_moe_route_ex(stream, logits, bias, T, E, n_group, topk_group, topk, route_scale, topk_idx, topk_w,
                             0u);
}

static beam_status router_sigmoid_call(beam_stream_t stream, const float* z, float* s, int64_t count, int fast) {
    if (count < 0 || count > (int64_t(1) << 40)) return BEAM_ERR_SHAPE;
    if (count == 0) return BEAM_OK;
    if (!z || !s) return BEAM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(z) & 3u) || (reinterpret_cast<uintptr_t>(s) & 3u)) return BEAM_ERR_ALIGN;
    const size_t nb = (size_t)count * 4u;
    if ((const void*)z != (const void*)s && overlaps(z, nb, s, nb)) return BEAM_ERR_ALIAS;
    DeviceInfo* info = nullptr;
    beam_status st = current_device(&info);
    if (st != BEAM_OK) return st;
    int64_t blocks = (count + 255) / 256;
    const int64_t cap = (int64_t)info->sms * 8;  // grid-stride beyond 8 blocks per SM
    if (blocks > cap) blocks = cap;
    beam::router_sigmoid_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(z, s, count,
                                                                                                    fast);
    if (cudaGetLastError() != cudaSuccess) return BEAM_ERR_CUDA;
    return BEAM_OK;
}

beam_status beam_router_sigmoid(beam_stream_t stream, const float* z, float* s, int64_t count) {
    return router_sigmoid_call(stream, z, s, count, 0);
}

beam_status beam_router_sigmoid_fast(beam_stream_t stream, const float* z, float* s, int64_t count) {
    return router_sigmoid_call(stream, z, s, count, 1);
}

beam_status beam_moe_combine_boundary(beam_stream_t stream, uint16_t* h, const uint16_t* expert_out,
                                      const float* topk_w, const uint16_t* post_w, const uint16_t* pre_w, int n,
                                      float eps, int64_t T, int D, uint16_t* y_out) {
    return beam_moe_combine_boundary_ex(stream, h, expert_out, topk_w, post_w, pre_w, n, eps, T, D, y_out,
                                        nullptr);
}

beam_status beam_qk_norm_ex(beam_stream_t stream, uint16_t* q, uint16_t* k, const uint16_t* q_w,
                            const uint16_t* k_w, const int32_t* pos, const float* rope_table, int64_t max_pos,
                            int64_t T, int n_q_heads, int n_kv_heads, int head_dim, float eps, int mode,
                            uint32_t flags) {
    if (T < 0 || T > (int64_t(1) << 40) || head_dim != BEAM_QK_HEAD_DIM || n_q_heads < 0 || n_kv_heads < 0 ||
        n_q_heads + n_kv_heads > 4096)
        return BEAM_ERR_SHAPE;
    if ((mode != BEAM_QK_ROPE && mode != BEAM_QK_SSMAX) || !(eps >= 0.0f) || !std::isfinite(eps) ||
        (mode == BEAM_QK_ROPE && max_pos < 1) || (flags & ~(BEAM_OPT_FORCE_EXACT_SUM | BEAM_OPT_PDL)))
        return BEAM_ERR_ARG;
    if (T == 0 || n_q_heads + n_kv_heads == 0) return BEAM_OK;
    if ((n_q_heads && !q) || (n_kv_heads && !k) || !q_w || !k_w || !pos || (mode == BEAM_QK_ROPE && !rope_table))
        return BEAM_ERR_NULL;
    if ((q && !aligned16(q)) || (k && !aligned16(k)) || !aligned16(q_w) || !aligned16(k_w) ||
        (reinterpret_cast<uintptr_t>(pos) & 3u) || (mode == BEAM_QK_ROPE && !aligned16(rope_table)))
        return BEAM_ERR_ALIGN;
    const size_t qb = (size_t)T * n_q_heads * head_dim * 2u, kb = (size_t)T * n_kv_heads * head_dim * 2u;
    const size_t wb = (size_t)head_dim * 2u, pb = (size_t)T * 4u;
    const size_t tb = mode == BEAM_QK_ROPE ? (size_t)max_pos * head_dim * 4u : 0u;
    if (overlaps(q, qb, k, kb) || overlaps(q, qb, q_w, wb) || overlaps(q, qb, k_w, wb) || overlaps(q, qb, pos, pb) ||
        overlaps(q, qb, rope_table, tb) || overlaps(k, kb, q_w, wb) || overlaps(k, kb, k_w, wb) ||
        overlaps(k, kb, pos, pb) || overlaps(k, kb, rope_table, tb))
        return BEAM_ERR_ALIAS;
    DeviceInfo* info = nullptr;
    beam_status st = current_device(&info);
    if (st != BEAM_OK) return st;
    beam::QKParams p;
    p.q = q;
    p.k = k;
    p.qw = q_w;
    p.kw = k_w;
    p.pos = pos;
    p.table = rope_table;
    p.max_pos = max_pos;
    p.T = T;
    p.nq = n_q_heads;
    p.nk = n_kv_heads;
    p.eps = eps;
    p.errk = error_factor_terms(8.0, 2 + 2);  // 8 terms per FP32 lane, 2 merges in the lane + 2 shuffle levels
    p.flags = (flags & BEAM_OPT_FORCE_EXACT_SUM) ? beam::kFlagForceExact : 0u;
    // one warp per token when there are enough tokens to fill the GPU (16
    // resident warps per SM); with fewer, up to one warp per 8-head batch of a token
    const int nbat = (n_q_heads + n_kv_heads + beam::kQKBatch - 1) / beam::kQKBatch;
    const int64_t target = (int64_t)info->sms * 16;
    int wpt = 1;
    if (T < target) {
        const int64_t want = (target + T - 1) / T;
        wpt = want < nbat ? (int)want : nbat;
    }
    p.batches_per_warp = (nbat + wpt - 1) / wpt;
    p.warps_per_token = (nbat + p.batches_per_warp - 1) / p.batches_per_warp;
    const int64_t blocks = (T * p.warps_per_token + 7) / 8;  // 8 warps per block
    if (blocks > 0x7FFFFFFF) return BEAM_ERR_SHAPE;
    const void* fn = mode == BEAM_QK_ROPE ? reinterpret_cast<const void*>(beam::qk_norm_kernel<0>)
                                          : reinterpret_cast<const void*>(beam::qk_norm_kernel<1>);
    void* args[] = {&p};
    if (flags & BEAM_OPT_PDL) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        cfg.stream = reinterpret_cast<cudaStream_t>(stream);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
            cudaGetLastError();
            return BEAM_ERR_CUDA;
        }
        return BEAM_OK;
    }
    if (cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(256), args, 0, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    return BEAM_OK;
}

beam_status beam_qk_norm(beam_stream_t stream, uint16_t* q, uint16_t* k, const uint16_t* q_w, const uint16_t* k_w,
                         const int32_t* pos, const float* rope_table, int64_t max_pos, int64_t T, int n_q_heads,
                         int n_kv_heads, int head_dim, float eps, int mode) {
    return beam_qk_norm_ex(stream, q, k, q_w, k_w, pos, rope_table, max_pos, T, n_q_heads, n_kv_heads, head_dim,
                           eps, mode, 0u);
}

beam_status beam_sync_status(beam_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    unsigned int word = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&word, beam::g_status_word, sizeof word, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(beam::g_status_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return BEAM_ERR_CUDA;
    }
    if (word & 1u) return BEAM_ERR_TIMEOUT;
    if (word & 2u) return BEAM_ERR_ARG;
    return BEAM_OK;
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
