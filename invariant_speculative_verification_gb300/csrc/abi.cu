// Host-side plumbing shared by every entry point: status strings, the
// thread-local last-error message, device queries and tensor-map encoding.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace spec {

static thread_local char g_last_error[512] = "";

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
}

spec_status fail(spec_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

spec_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return SPEC_OK;
    return fail(SPEC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base, const uint64_t *dims,
                  const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
        return false;
    }
    return true;
}

}  // namespace spec

extern "C" const char *spec_status_string(spec_status st) {
    switch (st) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    }
    return "SPEC_ERR_UNKNOWN";
}

extern "C" const char *spec_last_error(void) { return spec::g_last_error; }

// ---------------------------------------------------------------------------
// Test hook for the bounded-wait error path.  One thread arms an mbarrier for
// 16 transaction bytes and issues no copy, so the phase never completes and
// nothing is in flight; it then waits through the same bounded wait every
// kernel of the library uses, with `polls` polls, and reports
// SPEC_DEVERR_TIMEOUT when the wait runs out.  The kernel returns normally and
// the context stays usable.
// ---------------------------------------------------------------------------
namespace {
__global__ void wait_timeout_kernel(uint32_t polls, int32_t *dev_err) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    dev::mbar_init(&bar, 1);
    dev::fence_barrier_init();
    dev::mbar_arrive_expect_tx(&bar, 16);
    if (!dev::mbar_wait(&bar, 0, polls)) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
}
}  // namespace

extern "C" spec_status spec_debug_wait_timeout(uint32_t polls, int32_t *dev_err, spec_stream_t stream) {
    SPEC_CHECK_ARG(dev_err, "debug_wait_timeout: dev_err is NULL");
    SPEC_CHECK_ARG(polls >= 1 && polls <= (1u << 20), "debug_wait_timeout: polls must be in [1, 2^20] (polls=%u)",
                   polls);
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(polls, dev_err);
    return spec::cuda_status(cudaGetLastError(), "debug_wait_timeout launch");
}
