// dspark_fuse_ctx_noalloc: the fc context fusion without a caller workspace.
//
// The weight-streaming GEMM needs scratch memory for the partial sums of
// output tiles that several CTAs share, one counter per tile, and an error
// word. dspark_fuse_ctx takes that scratch from the caller's workspace; this
// variant keeps it in one fixed array of this library, so a caller that cannot
// allocate device memory can still run the fusion. Such callers include
// serving processes whose device memory is reserved up front by another
// allocator and has nothing left to hand out, latency-critical paths that may
// not call cudaMalloc (it can synchronise the whole device), and plugin hosts
// that do not let a library own device buffers.
//
// Limits: bs <= 2 (at most 14 activation rows, one 16-wide accumulator tile),
// at most 160 CTAs, at most 1024 output tiles of 128 channels (hidden <=
// 131072). The array is ~2.5 MiB and stays resident on every device that loads
// the library until the process exits.
#include <stddef.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "gemm.cuh"
#include "internal.h"

using namespace ds;

namespace {

constexpr int kNaBN = 16;
constexpr int kNaMaxCtas = 160;
constexpr int kNaMaxTiles = 1024;
constexpr int kNaMaxDevices = 64;
constexpr size_t kNaPartials = (size_t)2 * kNaMaxCtas * 128 * kNaBN;

struct NoAllocScratch {
    int err;
    int pad[63];
    int counters[kNaMaxTiles];
    float partials[kNaPartials];
};

// Scratch of the allocation-free fusion: shared by every call on a device.
static __device__ __align__(256) NoAllocScratch g_fc_scratch;

// Device address of g_fc_scratch, per device. The pointer is stored before the
// ready flag is raised (release), and read after the flag is seen (acquire), so
// a thread that finds the flag set also finds the pointer.
NoAllocScratch *g_dev_ptr[kNaMaxDevices];
std::atomic<bool> g_ready[kNaMaxDevices];
std::mutex g_setup_mu;

// Once per device, with that device current: resolve the array's device
// address and raise the kernel's shared-memory limit. Host threads that make
// their first call at the same time are serialised by the mutex.
dspark_status setup_device(int dev, NoAllocScratch **out) {
    if (dev < 0 || dev >= kNaMaxDevices) return DSPARK_ERR_UNSUPPORTED;
    if (!g_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_ready[dev].load(std::memory_order_relaxed)) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_fc_scratch) != cudaSuccess || ptr == nullptr) return DSPARK_ERR_CUDA;
            if (cudaFuncSetAttribute(gemm_swapab_kernel<kNaBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GemmCfg<kNaBN>::kSmemBytes) != cudaSuccess)
                return DSPARK_ERR_CUDA;
            g_dev_ptr[dev] = (NoAllocScratch *)ptr;
            g_ready[dev].store(true, std::memory_order_release);
        }
    }
    *out = g_dev_ptr[dev];
    return DSPARK_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" dspark_status dspark_fuse_ctx_noalloc(dspark_handle_t *h, const void *aux, float *x, int bs,
                                                 void *stream) {
    if (!h || !aux || !x) return DSPARK_ERR_NULL;
    // Only bf16 fc weights: the handle encodes the bf16 weight descriptor this
    // kernel reads for that format alone. Checked before any CUDA call.
    if (handle_geom(h)->weight_format != DSPARK_FMT_BF16) return DSPARK_ERR_UNSUPPORTED;
    if (!aligned16(aux) || !aligned16(x)) return DSPARK_ERR_ALIGN;
    if (bs <= 0 || 7 * bs > kNaBN) return DSPARK_ERR_SHAPE;
    const dspark_geom_t &g = *handle_geom(h);
    const int M = g.block * bs;
    if (M > kNaBN) return DSPARK_ERR_SHAPE;
    const int tiles = (g.hidden + 127) / 128;
    if (tiles > kNaMaxTiles) return DSPARK_ERR_SHAPE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    NoAllocScratch *s = nullptr;
    const dspark_status st = setup_device(dev, &s);
    if (st != DSPARK_OK) return st;
    cudaStream_t strm = (cudaStream_t)stream;
    // the tile counters must start at zero (a previous call may have stopped
    // early); the error word is kept until noalloc_check reads it
    if (cudaMemsetAsync(s->counters, 0, sizeof(s->counters), strm) != cudaSuccess) return DSPARK_ERR_CUDA;
    CUtensorMap b_aux;
    if (!encode_bf16_map(&b_aux, aux, M, (uint64_t)g.n_aux * g.hidden, kNaBN)) return DSPARK_ERR_CUDA;
    GemmParams p;
    memset(&p, 0, sizeof(p));
    p.n_out = g.hidden;
    p.K = g.n_aux * g.hidden;
    p.M = M;
    p.KB = (p.K + 63) / 64;
    p.tiles = tiles;
    p.units = (long long)p.tiles * p.KB;
    long long grid = p.units / 4;
    const int sms = handle_num_sms(h);
    if (grid > sms) grid = sms;
    if (grid > kNaMaxCtas) grid = kNaMaxCtas;
    if (grid < 1) grid = 1;
    p.grid = (int)grid;
    p.paired = 0;
    p.epi = EPI_STORE;
    p.out_f32 = x;
    p.ldo = g.hidden;
    p.partials = s->partials;
    p.counters = s->counters;
    p.err = &s->err;
    const CUtensorMap &a = *handle_fc_map(h);
    gemm_swapab_kernel<kNaBN><<<p.grid, 192, GemmCfg<kNaBN>::kSmemBytes, strm>>>(a, a, b_aux, p);
    return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

namespace ds {

// The error word of the fixed scratch on the current device: synchronise the
// stream, read it and clear it (DSPARK_OK when the no-alloc fusion has not run
// on this device yet).
dspark_status noalloc_check(void *stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (dev < 0 || dev >= kNaMaxDevices || !g_ready[dev].load(std::memory_order_acquire)) return DSPARK_OK;
    cudaStream_t strm = (cudaStream_t)stream;
    if (cudaStreamSynchronize(strm) != cudaSuccess) return DSPARK_ERR_CUDA;
    int *errp = &g_dev_ptr[dev]->err;
    int err = 0;
    if (cudaMemcpy(&err, errp, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (err && cudaMemset(errp, 0, sizeof(int)) != cudaSuccess) return DSPARK_ERR_CUDA;
    return (dspark_status)err;
}

}  // namespace ds
