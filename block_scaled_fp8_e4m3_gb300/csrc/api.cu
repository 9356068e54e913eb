// api.cu -- the extern "C" entry points declared in include/fp8bs.h.
//
// Each call validates every argument on the host, then enqueues kernels on
// the caller's stream.  Nothing is enqueued when validation fails.  The only
// device memory the library owns is one StatusBlock per device.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"

using namespace fp8bs;

namespace {

thread_local std::string g_last_error = "no error";

fp8_status fail(fp8_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

fp8_status cuda_fail(cudaError_t e, const char* where) {
    return fail(FP8_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
StatusBlock* g_status[kMaxDevices] = {};

// The current device's status block, allocated and zeroed on first use.
StatusBlock* status_block(fp8_status* err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = cuda_fail(e, "cudaGetDevice");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (g_status[dev] == nullptr) {
        void* p = nullptr;
        e = cudaMalloc(&p, sizeof(StatusBlock));
        if (e != cudaSuccess) {
            *err = cuda_fail(e, "cudaMalloc(status block)");
            return nullptr;
        }
        e = cudaMemset(p, 0, sizeof(StatusBlock));
        if (e != cudaSuccess) {
            cudaFree(p);
            *err = cuda_fail(e, "cudaMemset(status block)");
            return nullptr;
        }
        g_status[dev] = static_cast<StatusBlock*>(p);
    }
    *err = FP8_OK;
    return g_status[dev];
}

// Installs share per-device state on the GPU: the status block's checksum
// accumulator, verdict and grid-barrier counter (fp8_sync_install), or the
// static scratch (fp8_sync_install_noalloc).  Two installs that overlapped on
// the device -- issued on different streams or from different host threads --
// would corrupt each other's verdict, so every install is ordered after the
// previous one on the device: its stream waits on one event per device, which
// it then records.  Inside a stream capture the ordering is left to the
// caller (a capture cannot wait on an event recorded outside it).
class InstallOrder {
  public:
    explicit InstallOrder(cudaStream_t s) : lock_(mu_), s_(s) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaGetDevice(&dev_) != cudaSuccess || dev_ < 0 || dev_ >= kMaxDevices ||
            cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
            (void)cudaGetLastError();
            dev_ = -1;
            return;
        }
        if (ev_[dev_] == nullptr && cudaEventCreateWithFlags(&ev_[dev_], cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            ev_[dev_] = nullptr;
            dev_ = -1;
            return;
        }
        if (used_[dev_]) err_ = cudaStreamWaitEvent(s, ev_[dev_], 0);
    }
    ~InstallOrder() {
        if (dev_ >= 0 && cudaEventRecord(ev_[dev_], s_) == cudaSuccess) used_[dev_] = true;
    }
    cudaError_t error() const { return err_; }

  private:
    static std::mutex mu_;
    static cudaEvent_t ev_[kMaxDevices];
    static bool used_[kMaxDevices];
    std::lock_guard<std::mutex> lock_;
    cudaStream_t s_;
    int dev_ = -1;
    cudaError_t err_ = cudaSuccess;
};
std::mutex InstallOrder::mu_;
cudaEvent_t InstallOrder::ev_[kMaxDevices] = {};
bool InstallOrder::used_[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

fp8_status check_out(const fp8_tensor* t, const char* name, int recipe, int layout, int64_t rows, int64_t cols,
                     bool need_scales = true) {
    if (t == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s is NULL", name);
    const bool empty = rows == 0 || cols == 0;  // empty tensors may carry NULL pointers
    if (!empty && (t->codes == nullptr || (need_scales && t->scales == nullptr)))
        return fail(FP8_ERR_INVALID_ARG, "%s: codes/scales pointer is NULL", name);
    if (t->recipe != recipe) return fail(FP8_ERR_INVALID_ARG, "%s: recipe %d, expected %d", name, t->recipe, recipe);
    if (t->layout != layout) return fail(FP8_ERR_INVALID_ARG, "%s: layout %d, expected %d", name, t->layout, layout);
    if (t->rows != rows || t->cols != cols)
        return fail(FP8_ERR_INVALID_ARG, "%s: shape %lldx%lld, expected %lldx%lld", name, (long long)t->rows,
                    (long long)t->cols, (long long)rows, (long long)cols);
    if (!aligned16(t->codes) || (need_scales && !aligned16(t->scales)))
        return fail(FP8_ERR_ALIGNMENT, "%s: codes/scales not 16-byte aligned", name);
    return FP8_OK;
}

fp8_status check_input(const void* x, int64_t rows, int64_t cols, int64_t ld, const char* name) {
    if (rows < 0 || cols < 0) return fail(FP8_ERR_INVALID_ARG, "%s: negative size", name);
    if (rows > 0 && cols > 0 && x == nullptr) return fail(FP8_ERR_INVALID_ARG, "%s is NULL", name);
    if (ld < cols) return fail(FP8_ERR_INVALID_ARG, "%s: ld %lld < cols %lld", name, (long long)ld, (long long)cols);
    if (!aligned16(x) || (ld % 8) != 0) return fail(FP8_ERR_ALIGNMENT, "%s: not 16-byte aligned or ld %% 8 != 0", name);
    if (rows > (int64_t)INT32_MAX || cols > (int64_t)INT32_MAX)
        return fail(FP8_ERR_UNSUPPORTED, "%s: dimension above 2^31-1", name);
    return FP8_OK;
}

int64_t mx_scale_bytes(int64_t rows, int64_t cols) { return cdiv(rows, 128) * cdiv(cols, 128) * 512; }

// ---------------------------------------------------------------- sync layout
constexpr uint64_t kSyncMagic = 0x31434E5953385046ull;  // bytes "FP8SYNC1"
constexpr uint32_t kSyncVersion = 2;                     // the NH checksum
constexpr uint64_t kHeaderBytes = 64, kEntryBytes = 128;

uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

// The checksum term of payload word w at word index i (format version 2):
// ((lo + i K1) mod 2^32) * ((hi + i K2) mod 2^32), summed mod 2^64.
uint64_t word_term(uint64_t w, uint64_t i) {
    const uint32_t a = (uint32_t)w + (uint32_t)i * 0x9E3779B9u;
    const uint32_t b = (uint32_t)(w >> 32) + (uint32_t)i * 0x85EBCA6Bu;
    return (uint64_t)a * b;
}

struct EntryLayout {
    uint64_t data_off, data_bytes, scale_off, scale_bytes;
};

fp8_status entry_bytes(const fp8_sync_entry& e, int i, uint64_t* db, uint64_t* sb) {
    const fp8_tensor& t = e.t;
    if (e.reserved != 0) return fail(FP8_ERR_INVALID_ARG, "entry %d: reserved field must be 0", i);
    if (t.rows < 0 || t.cols < 0) return fail(FP8_ERR_INVALID_ARG, "entry %d: negative shape", i);
    if (t.codes == nullptr && t.rows * t.cols > 0) return fail(FP8_ERR_INVALID_ARG, "entry %d: data is NULL", i);
    if (!aligned16(t.codes)) return fail(FP8_ERR_ALIGNMENT, "entry %d: data not 16-byte aligned", i);
    if (e.kind == FP8_SYNC_BF16) {
        if (t.recipe != 0 || t.layout != 0 || t.scales != nullptr)
            return fail(FP8_ERR_INVALID_ARG, "entry %d: bf16 entry with recipe/layout/scales", i);
        *db = (uint64_t)(t.rows * t.cols * 2);
        *sb = 0;
        return FP8_OK;
    }
    if (e.kind != FP8_SYNC_FP8) return fail(FP8_ERR_INVALID_ARG, "entry %d: unknown kind %d", i, e.kind);
    if (t.scales == nullptr || !aligned16(t.scales))
        return fail(FP8_ERR_ALIGNMENT, "entry %d: scales NULL or not 16-byte aligned", i);
    *db = (uint64_t)(t.rows * t.cols);
    if (t.recipe == FP8_RECIPE_BLOCKWISE_FP32 && t.layout == FP8_LAYOUT_GROUP_1x128 && t.cols % 128 == 0)
        *sb = (uint64_t)((t.cols / 128) * t.rows * 4);
    else if (t.recipe == FP8_RECIPE_BLOCKWISE_FP32 && t.layout == FP8_LAYOUT_BLOCK_128x128 && t.rows % 128 == 0 &&
             t.cols % 128 == 0)
        *sb = (uint64_t)((t.rows / 128) * (t.cols / 128) * 4);
    else if ((t.recipe == FP8_RECIPE_MXFP8 || t.recipe == FP8_RECIPE_BLOCKWISE_POW2) &&
             t.layout == FP8_LAYOUT_MX_1x32 && t.cols % 32 == 0)
        *sb = (uint64_t)mx_scale_bytes(t.rows, t.cols);
    else
        return fail(FP8_ERR_UNSUPPORTED, "entry %d: recipe %d / layout %d / shape %lldx%lld cannot be synced", i,
                    t.recipe, t.layout, (long long)t.rows, (long long)t.cols);
    return FP8_OK;
}

fp8_status sync_layout(const fp8_sync_entry* e, int32_t n, std::vector<EntryLayout>* lay, uint64_t* total) {
    if (n < 0 || (n > 0 && e == nullptr)) return fail(FP8_ERR_INVALID_ARG, "bad entry list");
    lay->resize((size_t)n);
    uint64_t off = round_up(kHeaderBytes + kEntryBytes * (uint64_t)n, 256);
    for (int32_t i = 0; i < n; ++i) {
        uint64_t db, sb;
        fp8_status s = entry_bytes(e[i], i, &db, &sb);
        if (s != FP8_OK) return s;
        EntryLayout& L = (*lay)[(size_t)i];
        L.data_off = off;
        L.data_bytes = db;
        off = round_up(off + db, 256);
        L.scale_off = sb ? off : 0;
        L.scale_bytes = sb;
        off = round_up(off + sb, 256);
    }
    *total = off;
    return FP8_OK;
}

void put64(uint8_t* p, uint64_t v) {
    for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
void put32(uint8_t* p, uint32_t v) {
    for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
uint64_t get64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
    return v;
}
uint32_t get32(const uint8_t* p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

// Header + entry table (+ zero padding up to the first segment) as the
// payload must hold them; checksum field left 0.
std::vector<uint8_t> build_table(const fp8_sync_entry* e, int32_t n, const std::vector<EntryLayout>& lay,
                                 uint64_t total) {
    const uint64_t data_offset = round_up(kHeaderBytes + kEntryBytes * (uint64_t)n, 256);
    std::vector<uint8_t> h((size_t)data_offset, 0);
    put64(&h[0], kSyncMagic);
    put32(&h[8], kSyncVersion);
    put32(&h[12], (uint32_t)n);
    put64(&h[16], total);
    put64(&h[24], data_offset);
    for (int32_t i = 0; i < n; ++i) {
        uint8_t* t = &h[(size_t)(kHeaderBytes + kEntryBytes * (uint64_t)i)];
        put64(t + 0, e[i].tag);
        put32(t + 8, (uint32_t)e[i].kind);
        put32(t + 12, (uint32_t)e[i].t.recipe);
        put64(t + 16, (uint64_t)e[i].t.rows);
        put64(t + 24, (uint64_t)e[i].t.cols);
        put32(t + 32, (uint32_t)e[i].t.layout);
        put64(t + 40, lay[(size_t)i].data_off);
        put64(t + 48, lay[(size_t)i].data_bytes);
        put64(t + 56, lay[(size_t)i].scale_off);
        put64(t + 64, lay[(size_t)i].scale_bytes);
    }
    return h;
}

uint64_t table_checksum(const std::vector<uint8_t>& h) {
    uint64_t sum = 0;
    for (uint64_t i = kHeaderBytes / 8; i < h.size() / 8; ++i) sum += word_term(get64(&h[(size_t)(8 * i)]), i);
    return sum;
}


// ---------------------------------------------------------------- install without allocation
// For callers that cannot allocate device memory: the checksum accumulator,
// the verdict and the segment table of fp8_sync_install_noalloc live in this
// file-scope device array instead of the per-device block the library would
// otherwise cudaMalloc.  Every GPU that loads the library holds it until the
// process exits.  All calls share it, so calls that overlap on the GPU race.
constexpr int kNoAllocMaxEntries = 128;
constexpr int kNoAllocMaxSegs = 2 * kNoAllocMaxEntries;
constexpr uint64_t kNoAllocTableBytes = (kHeaderBytes + kEntryBytes * kNoAllocMaxEntries + 255) / 256 * 256;

struct NoAllocScratch {
    StatusBlock status;
    CopySeg segs[kNoAllocMaxSegs];
};

static __device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocScratch)];

std::mutex g_noalloc_mu;
NoAllocScratch* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once
// per device; in host code the array's name is only a stand-in).
NoAllocScratch* noalloc_scratch(fp8_status* err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = cuda_fail(e, "cudaGetDevice");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            *err = cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
            return nullptr;
        }
        g_noalloc_ptr[dev] = static_cast<NoAllocScratch*>(ptr);
    }
    *err = FP8_OK;
    return g_noalloc_ptr[dev];
}

// Scatter variant that reads its segment table and the verify kernel's
// verdict from the scratch array; all segments in one launch.
__global__ void __launch_bounds__(256) k_sync_scatter_table(const NoAllocScratch* sc, int nseg) {
    if (*reinterpret_cast<const volatile unsigned int*>(&sc->status.verdict) != 0) return;
    __shared__ uint64_t start[kNoAllocMaxSegs + 1];
    if (threadIdx.x == 0) {
        uint64_t acc = 0;
        for (int i = 0; i < nseg; ++i) {
            start[i] = acc;
            acc += (sc->segs[i].bytes + 15) / 16;
        }
        start[nseg] = acc;
    }
    __syncthreads();
    const uint64_t chunks = start[nseg];
    for (uint64_t c = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; c < chunks;
         c += (uint64_t)gridDim.x * blockDim.x) {
        int lo = 0, hi = nseg;  // start[lo] <= c < start[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (start[mid] <= c) lo = mid; else hi = mid;
        }
        const CopySeg sg = sc->segs[lo];
        const uint64_t off = (c - start[lo]) * 16;
        const uint4 v = *reinterpret_cast<const uint4*>(sg.src + off);
        if (off + 16 <= sg.bytes) {
            *reinterpret_cast<uint4*>(sg.dst + off) = v;
        } else {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            for (uint64_t b = 0; off + b < sg.bytes; ++b) sg.dst[off + b] = (uint8_t)(w[b / 4] >> (8 * (b % 4)));
        }
    }
}

// Header + entry table into a caller-provided buffer (no allocation).
void fill_table(uint8_t* h, uint64_t data_offset, const fp8_sync_entry* e, int32_t n, const EntryLayout* lay,
                uint64_t total) {
    memset(h, 0, (size_t)data_offset);
    put64(&h[0], kSyncMagic);
    put32(&h[8], kSyncVersion);
    put32(&h[12], (uint32_t)n);
    put64(&h[16], total);
    put64(&h[24], data_offset);
    for (int32_t i = 0; i < n; ++i) {
        uint8_t* t = &h[(size_t)(kHeaderBytes + kEntryBytes * (uint64_t)i)];
        put64(t + 0, e[i].tag);
        put32(t + 8, (uint32_t)e[i].kind);
        put32(t + 12, (uint32_t)e[i].t.recipe);
        put64(t + 16, (uint64_t)e[i].t.rows);
        put64(t + 24, (uint64_t)e[i].t.cols);
        put32(t + 32, (uint32_t)e[i].t.layout);
        put64(t + 40, lay[i].data_off);
        put64(t + 48, lay[i].data_bytes);
        put64(t + 56, lay[i].scale_off);
        put64(t + 64, lay[i].scale_bytes);
    }
}

}  // namespace

// ===========================================================================
extern "C" {

int32_t fp8_abi_version(void) { return FP8BS_ABI_VERSION; }

const char* fp8_last_error(void) { return g_last_error.c_str(); }

int64_t fp8_mx_scale_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return 0;
    return mx_scale_bytes(rows, cols);
}

int64_t fp8_mx_grouped_scale_bytes(int64_t total_rows, int64_t cols, int32_t num_groups) {
    if (total_rows < 0 || cols < 0 || num_groups < 0) return 0;
    return (cdiv(total_rows, 128) + num_groups) * cdiv(cols, 128) * 512;
}

fp8_status fp8_quantize_group(const void* x_bf16, int64_t M, int64_t K, int64_t ld, fp8_axis axis,
                              const fp8_tensor* out, fp8_stream_t stream) {
    fp8_status s = check_input(x_bf16, M, K, ld, "x");
    if (s != FP8_OK) return s;
    if (axis == FP8_AXIS_K) {
        if (K % 128 != 0) return fail(FP8_ERR_UNSUPPORTED, "1x128 groups need K %% 128 == 0 (K = %lld)", (long long)K);
        const bool pow2 = out != nullptr && out->recipe == FP8_RECIPE_BLOCKWISE_POW2;
        s = pow2 ? check_out(out, "out", FP8_RECIPE_BLOCKWISE_POW2, FP8_LAYOUT_MX_1x32, M, K)
                 : check_out(out, "out", FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, M, K);
        if (s != FP8_OK) return s;
        cudaError_t e = launch_quant_group_k(static_cast<const uint16_t*>(x_bf16), M, K, ld,
                                             static_cast<uint8_t*>(out->codes), out->scales, pow2,
                                             reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? FP8_OK : cuda_fail(e, "quantize_group(K)");
    }
    if (axis == FP8_AXIS_M) {
        if (M % 128 != 0 || K % 8 != 0)
            return fail(FP8_ERR_UNSUPPORTED, "128x1 groups need M %% 128 == 0 and K %% 8 == 0 (M = %lld, K = %lld)",
                        (long long)M, (long long)K);
        const bool pow2 = out != nullptr && out->recipe == FP8_RECIPE_BLOCKWISE_POW2;
        s = pow2 ? check_out(out, "out", FP8_RECIPE_BLOCKWISE_POW2, FP8_LAYOUT_MX_1x32, K, M)
                 : check_out(out, "out", FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, K, M);
        if (s != FP8_OK) return s;
        cudaError_t e = launch_quant_group_m(static_cast<const uint16_t*>(x_bf16), M, K, ld,
                                             static_cast<uint8_t*>(out->codes), out->scales, pow2,
                                             reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? FP8_OK : cuda_fail(e, "quantize_group(M)");
    }
    return fail(FP8_ERR_INVALID_ARG, "unknown axis %d", (int)axis);
}

fp8_status fp8_requantize_transposed(const fp8_tensor* in, const fp8_tensor* out, fp8_stream_t stream) {
    if (in == nullptr || out == nullptr) return fail(FP8_ERR_INVALID_ARG, "NULL argument");
    const int64_t M = in->rows, K = in->cols;
    if (M < 0 || K < 0) return fail(FP8_ERR_INVALID_ARG, "negative size");
    if (M % 128 != 0 || K % 128 != 0)
        return fail(FP8_ERR_UNSUPPORTED, "requantize_transposed needs M, K multiples of 128 (M = %lld, K = %lld)",
                    (long long)M, (long long)K);
    fp8_status s = check_out(in, "in", FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, M, K);
    if (s != FP8_OK) return s;
    s = check_out(out, "out", FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, K, M);
    if (s != FP8_OK) return s;
    cudaError_t e = launch_requant_group_m(static_cast<const uint8_t*>(in->codes), static_cast<const float*>(in->scales),
                                           M, K, static_cast<uint8_t*>(out->codes), static_cast<float*>(out->scales),
                                           reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "requantize_transposed");
}

fp8_status fp8_quantize_block(const void* w_bf16, int64_t N, int64_t K, int64_t ld, const fp8_tensor* out,
                              const fp8_tensor* out_t, fp8_stream_t stream) {
    fp8_status s = check_input(w_bf16, N, K, ld, "w");
    if (s != FP8_OK) return s;
    if (N % 128 != 0 || K % 128 != 0)
        return fail(FP8_ERR_UNSUPPORTED, "128x128 blocks need N, K multiples of 128 (N = %lld, K = %lld)", (long long)N,
                    (long long)K);
    const bool pow2 = out != nullptr && out->recipe == FP8_RECIPE_BLOCKWISE_POW2;
    const int recipe = pow2 ? FP8_RECIPE_BLOCKWISE_POW2 : FP8_RECIPE_BLOCKWISE_FP32;
    const int layout = pow2 ? FP8_LAYOUT_MX_1x32 : FP8_LAYOUT_BLOCK_128x128;
    s = check_out(out, "out", recipe, layout, N, K);
    if (s != FP8_OK) return s;
    if (out_t != nullptr) {
        s = check_out(out_t, "out_t", recipe, layout, K, N);
        if (s != FP8_OK) return s;
    }
    cudaError_t e = launch_quant_block(static_cast<const uint16_t*>(w_bf16), N, K, ld, static_cast<uint8_t*>(out->codes),
                                       out->scales, out_t ? static_cast<uint8_t*>(out_t->codes) : nullptr,
                                       out_t ? out_t->scales : nullptr, pow2, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "quantize_block");
}

fp8_status fp8_param_requantize(float* master, const float* delta, int64_t N, int64_t K, int64_t ld,
                                const fp8_tensor* out, const fp8_tensor* out_t, fp8_stream_t stream) {
    if (N < 0 || K < 0) return fail(FP8_ERR_INVALID_ARG, "master: negative size");
    if (N > 0 && K > 0 && master == nullptr) return fail(FP8_ERR_INVALID_ARG, "master is NULL");
    if (ld < K) return fail(FP8_ERR_INVALID_ARG, "master: ld %lld < cols %lld", (long long)ld, (long long)K);
    if (!aligned16(master) || !aligned16(delta) || (ld % 4) != 0)
        return fail(FP8_ERR_ALIGNMENT, "master/delta: not 16-byte aligned or ld %% 4 != 0");
    if (N > (int64_t)INT32_MAX || K > (int64_t)INT32_MAX)
        return fail(FP8_ERR_UNSUPPORTED, "master: dimension above 2^31-1");
    if (N % 128 != 0 || K % 128 != 0)
        return fail(FP8_ERR_UNSUPPORTED, "128x128 blocks need N, K multiples of 128 (N = %lld, K = %lld)", (long long)N,
                    (long long)K);
    const bool pow2 = out != nullptr && out->recipe == FP8_RECIPE_BLOCKWISE_POW2;
    const int recipe = pow2 ? FP8_RECIPE_BLOCKWISE_POW2 : FP8_RECIPE_BLOCKWISE_FP32;
    const int layout = pow2 ? FP8_LAYOUT_MX_1x32 : FP8_LAYOUT_BLOCK_128x128;
    fp8_status s = check_out(out, "out", recipe, layout, N, K);
    if (s != FP8_OK) return s;
    if (out_t != nullptr) {
        s = check_out(out_t, "out_t", recipe, layout, K, N);
        if (s != FP8_OK) return s;
    }
    cudaError_t e = launch_param_requant(master, delta, N, K, ld, static_cast<uint8_t*>(out->codes), out->scales,
                                         out_t ? static_cast<uint8_t*>(out_t->codes) : nullptr,
                                         out_t ? out_t->scales : nullptr, pow2, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "param_requantize");
}

namespace {
// The activation recipes of the fused producers: out->recipe picks the
// layout; returns the kernel's recipe index or -1.
int activation_recipe(const fp8_tensor* out, int* layout) {
    if (out == nullptr) return -1;
    switch (out->recipe) {
        case FP8_RECIPE_BLOCKWISE_FP32: *layout = FP8_LAYOUT_GROUP_1x128; return 0;
        case FP8_RECIPE_BLOCKWISE_POW2: *layout = FP8_LAYOUT_MX_1x32; return 1;
        case FP8_RECIPE_MXFP8: *layout = FP8_LAYOUT_MX_1x32; return 2;
        default: return -1;
    }
}

fp8_status check_bf16_out(const void* y, int64_t cols, int64_t ldy, const char* name) {
    if (y == nullptr) return FP8_OK;
    if (ldy < cols) return fail(FP8_ERR_INVALID_ARG, "%s: ld %lld < cols %lld", name, (long long)ldy, (long long)cols);
    if (!aligned16(y) || ldy % 8 != 0) return fail(FP8_ERR_ALIGNMENT, "%s: not 16-byte aligned or ld %% 8 != 0", name);
    return FP8_OK;
}
}  // namespace

fp8_status fp8_rmsnorm_quantize(const void* x_bf16, const void* gamma_bf16, int64_t M, int64_t K, int64_t ld,
                                float eps, void* y_bf16, int64_t ldy, float* rstd, const fp8_tensor* out,
                                fp8_stream_t stream) {
    fp8_status s = check_input(x_bf16, M, K, ld, "x");
    if (s != FP8_OK) return s;
    if (K % 128 != 0 || K == 0 || K > 8192)
        return fail(FP8_ERR_UNSUPPORTED, "rmsnorm_quantize needs K %% 128 == 0 and 0 < K <= 8192 (K = %lld)",
                    (long long)K);
    if (gamma_bf16 == nullptr || !aligned16(gamma_bf16)) return fail(FP8_ERR_ALIGNMENT, "gamma NULL or misaligned");
    if (!(eps >= 0.0f) || eps > 3.402823466e38f) return fail(FP8_ERR_INVALID_ARG, "eps must be finite and >= 0");
    s = check_bf16_out(y_bf16, K, ldy, "y");
    if (s != FP8_OK) return s;
    if (reinterpret_cast<uintptr_t>(rstd) & 3u) return fail(FP8_ERR_ALIGNMENT, "rstd misaligned");
    int layout = 0;
    const int rec = activation_recipe(out, &layout);
    if (rec < 0) return fail(FP8_ERR_INVALID_ARG, "out: NULL or unsupported recipe");
    s = check_out(out, "out", out->recipe, layout, M, K);
    if (s != FP8_OK) return s;
    cudaError_t e = launch_rmsnorm_quant(static_cast<const uint16_t*>(x_bf16), static_cast<const uint16_t*>(gamma_bf16),
                                         M, K, ld, eps, static_cast<uint16_t*>(y_bf16), ldy, rstd,
                                         static_cast<uint8_t*>(out->codes), out->scales, rec,
                                         reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "rmsnorm_quantize");
}

fp8_status fp8_swiglu_quantize(const void* gu_bf16, int64_t M, int64_t F, int64_t ld, void* h_bf16, int64_t ldh,
                               const fp8_tensor* out, fp8_stream_t stream) {
    if (F < 0 || F > (int64_t)INT32_MAX / 2) return fail(FP8_ERR_INVALID_ARG, "gu: bad F");
    fp8_status s = check_input(gu_bf16, M, 2 * F, ld, "gu");
    if (s != FP8_OK) return s;
    if (F % 128 != 0) return fail(FP8_ERR_UNSUPPORTED, "swiglu_quantize needs F %% 128 == 0 (F = %lld)", (long long)F);
    s = check_bf16_out(h_bf16, F, ldh, "h");
    if (s != FP8_OK) return s;
    int layout = 0;
    const int rec = activation_recipe(out, &layout);
    if (rec < 0) return fail(FP8_ERR_INVALID_ARG, "out: NULL or unsupported recipe");
    s = check_out(out, "out", out->recipe, layout, M, F);
    if (s != FP8_OK) return s;
    if (F == 0) return FP8_OK;
    cudaError_t e = launch_swiglu_quant(static_cast<const uint16_t*>(gu_bf16), M, F, ld, static_cast<uint16_t*>(h_bf16),
                                        ldh, static_cast<uint8_t*>(out->codes), out->scales, rec,
                                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "swiglu_quantize");
}

fp8_status fp8_quantize_mx(const void* x_bf16, int64_t R, int64_t K, int64_t ld, const fp8_tensor* out,
                           fp8_stream_t stream) {
    fp8_status s = check_input(x_bf16, R, K, ld, "x");
    if (s != FP8_OK) return s;
    if (K % 32 != 0) return fail(FP8_ERR_UNSUPPORTED, "1x32 blocks need K %% 32 == 0 (K = %lld)", (long long)K);
    s = check_out(out, "out", FP8_RECIPE_MXFP8, FP8_LAYOUT_MX_1x32, R, K);
    if (s != FP8_OK) return s;
    cudaError_t e = launch_quant_mx(static_cast<const uint16_t*>(x_bf16), R, K, ld, static_cast<uint8_t*>(out->codes),
                                    static_cast<uint8_t*>(out->scales), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "quantize_mx");
}

fp8_status fp8_quantize_mx_transposed(const void* x_bf16, int64_t R, int64_t K, int64_t ld, const fp8_tensor* out,
                                      fp8_stream_t stream) {
    fp8_status s = check_input(x_bf16, R, K, ld, "x");
    if (s != FP8_OK) return s;
    if (R % 128 != 0 || K % 8 != 0)
        return fail(FP8_ERR_UNSUPPORTED, "32x1 blocks need R %% 128 == 0 and K %% 8 == 0 (R = %lld, K = %lld)",
                    (long long)R, (long long)K);
    s = check_out(out, "out", FP8_RECIPE_MXFP8, FP8_LAYOUT_MX_1x32, K, R);
    if (s != FP8_OK) return s;
    cudaError_t e = launch_quant_mx_t(static_cast<const uint16_t*>(x_bf16), R, K, ld, static_cast<uint8_t*>(out->codes),
                                      static_cast<uint8_t*>(out->scales), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "quantize_mx_transposed");
}

fp8_status fp8_permute_rows_mx(const fp8_tensor* src, const int32_t* gather_dev, const int32_t* m_offsets_dev,
                               int32_t num_groups, const fp8_tensor* dst, fp8_stream_t stream) {
    if (src == nullptr || dst == nullptr || gather_dev == nullptr || m_offsets_dev == nullptr)
        return fail(FP8_ERR_INVALID_ARG, "NULL argument");
    if (num_groups < 1 || num_groups > 1024) return fail(FP8_ERR_UNSUPPORTED, "num_groups must be in [1, 1024]");
    fp8_status s = check_out(src, "src", FP8_RECIPE_MXFP8, FP8_LAYOUT_MX_1x32, src->rows, src->cols);
    if (s != FP8_OK) return s;
    if (src->cols % 128 != 0 || src->rows < 0)
        return fail(FP8_ERR_UNSUPPORTED, "permute needs cols %% 128 == 0 (cols = %lld)", (long long)src->cols);
    s = check_out(dst, "dst", FP8_RECIPE_MXFP8, FP8_LAYOUT_MX_1x32_GROUPED, dst->rows, src->cols);
    if (s != FP8_OK) return s;
    if (!aligned16(gather_dev) || (reinterpret_cast<uintptr_t>(m_offsets_dev) & 3u))
        return fail(FP8_ERR_ALIGNMENT, "gather/m_offsets misaligned");
    fp8_status se;
    StatusBlock* st = status_block(&se);
    if (st == nullptr) return se;
    cudaError_t e = launch_permute_rows_mx(
        static_cast<const uint8_t*>(src->codes), static_cast<const uint8_t*>(src->scales), src->rows, src->cols,
        gather_dev, m_offsets_dev, num_groups, dst->rows, static_cast<uint8_t*>(dst->codes),
        static_cast<uint8_t*>(dst->scales), fp8_mx_grouped_scale_bytes(dst->rows, dst->cols, num_groups), st,
        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "permute_rows_mx");
}

fp8_status fp8_dispatch_quantize_mx(const void* x_bf16, int64_t T, int64_t K, int64_t ld, const int32_t* dst_index_dev,
                                    int32_t top_k, const int32_t* m_offsets_dev, int32_t num_groups,
                                    const fp8_tensor* dst, fp8_stream_t stream) {
    fp8_status s = check_input(x_bf16, T, K, ld, "x");
    if (s != FP8_OK) return s;
    if (dst == nullptr || m_offsets_dev == nullptr || (T > 0 && top_k > 0 && dst_index_dev == nullptr))
        return fail(FP8_ERR_INVALID_ARG, "NULL argument");
    if (num_groups < 1 || num_groups > 1024) return fail(FP8_ERR_UNSUPPORTED, "num_groups must be in [1, 1024]");
    if (top_k < 0 || top_k > 64) return fail(FP8_ERR_UNSUPPORTED, "top_k must be in [0, 64]");
    if (K % 128 != 0 || K == 0)
        return fail(FP8_ERR_UNSUPPORTED, "dispatch_quantize needs K %% 128 == 0 and K > 0 (K = %lld)", (long long)K);
    s = check_out(dst, "dst", FP8_RECIPE_MXFP8, FP8_LAYOUT_MX_1x32_GROUPED, dst->rows, K);
    if (s != FP8_OK) return s;
    if ((reinterpret_cast<uintptr_t>(dst_index_dev) & 3u) || (reinterpret_cast<uintptr_t>(m_offsets_dev) & 3u))
        return fail(FP8_ERR_ALIGNMENT, "dst_index/m_offsets misaligned");
    fp8_status se;
    StatusBlock* st = status_block(&se);
    if (st == nullptr) return se;
    cudaError_t e = launch_dispatch_quant_mx(
        static_cast<const uint16_t*>(x_bf16), T, K, ld, dst_index_dev, top_k, m_offsets_dev, num_groups, dst->rows,
        static_cast<uint8_t*>(dst->codes), static_cast<uint8_t*>(dst->scales),
        fp8_mx_grouped_scale_bytes(dst->rows, K, num_groups), st, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "dispatch_quantize_mx");
}

fp8_status fp8_gemm_blockscaled(const fp8_tensor* A, const fp8_tensor* B, void* D, int64_t ldd, int32_t d_dtype,
                                int32_t op, const fp8_tensor* d_quant, fp8_stream_t stream) {
    if (A == nullptr || B == nullptr) return fail(FP8_ERR_INVALID_ARG, "A or B is NULL");
    const int64_t M = A->rows, K = A->cols, N = B->rows;
    if (M < 0 || N < 0 || K < 0) return fail(FP8_ERR_INVALID_ARG, "negative size");
    if (B->cols != K) return fail(FP8_ERR_INVALID_ARG, "A has K = %lld, B has K = %lld", (long long)K, (long long)B->cols);
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return fail(FP8_ERR_UNSUPPORTED, "size too large");
    if (K % 128 != 0 || K == 0) return fail(FP8_ERR_UNSUPPORTED, "GEMM needs K %% 128 == 0 and K > 0 (K = %lld)", (long long)K);
    if (N % 16 != 0) return fail(FP8_ERR_UNSUPPORTED, "GEMM needs N %% 16 == 0 (N = %lld)", (long long)N);
    if (M > 0 && N > 0 && D == nullptr) return fail(FP8_ERR_INVALID_ARG, "D is NULL");
    if (!aligned16(D) || ldd < N || ldd % 8 != 0) return fail(FP8_ERR_ALIGNMENT, "D not 16-byte aligned or bad ldd");
    if (d_dtype != FP8_OUT_BF16 && d_dtype != FP8_OUT_F32) return fail(FP8_ERR_INVALID_ARG, "unknown d_dtype");
    if (d_dtype == FP8_OUT_F32 && (ldd % 4) != 0) return fail(FP8_ERR_ALIGNMENT, "bad ldd");
    fp8_status s;
    fp8_status se;
    StatusBlock* st = status_block(&se);
    if (st == nullptr) return se;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

    if (A->recipe == FP8_RECIPE_BLOCKWISE_FP32) {
        s = check_out(A, "A", FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, M, K);
        if (s != FP8_OK) return s;
        if (N % 128 != 0) return fail(FP8_ERR_UNSUPPORTED, "blockwise GEMM needs N %% 128 == 0 (N = %lld)", (long long)N);
        int sb_per_row;
        if (op == FP8_GEMM_FWD || op == FP8_GEMM_DGRAD) {
            s = check_out(B, "B", FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_BLOCK_128x128, N, K);
            sb_per_row = 0;
        } else if (op == FP8_GEMM_WGRAD) {
            s = check_out(B, "B", FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, N, K);
            sb_per_row = 1;
        } else {
            return fail(FP8_ERR_INVALID_ARG, "unknown op %d", op);
        }
        if (s != FP8_OK) return s;
        uint8_t* qc = nullptr;
        float* qs = nullptr;
        if (d_quant != nullptr) {
            if (d_dtype != FP8_OUT_BF16) return fail(FP8_ERR_INVALID_ARG, "fused quantization needs bf16 D");
            s = check_out(d_quant, "d_quant", FP8_RECIPE_BLOCKWISE_FP32, FP8_LAYOUT_GROUP_1x128, M, N);
            if (s != FP8_OK) return s;
            qc = static_cast<uint8_t*>(d_quant->codes);
            qs = static_cast<float*>(d_quant->scales);
        }
        GemmBlockwiseArgs a;
        a.a_codes = static_cast<const uint8_t*>(A->codes);
        a.b_codes = static_cast<const uint8_t*>(B->codes);
        a.sa = static_cast<const float*>(A->scales);
        a.sb = static_cast<const float*>(B->scales);
        a.sb_per_row = sb_per_row;
        a.M = M;
        a.N = N;
        a.K = K;
        a.D = D;
        a.ldd = ldd;
        a.d_f32 = d_dtype == FP8_OUT_F32;
        a.q_codes = qc;
        a.q_scales = qs;
        cudaError_t e = launch_gemm_blockwise(a, st, cs);
        return e == cudaSuccess ? FP8_OK : cuda_fail(e, "gemm_blockscaled(blockwise)");
    }
    if (A->recipe == FP8_RECIPE_MXFP8 || A->recipe == FP8_RECIPE_BLOCKWISE_POW2) {
        // both run on the block-scaled MMA; the power-of-two blockwise
        // recipe's scales are MX scales constant over each group
        const int recipe = A->recipe;
        const bool pow2 = recipe == FP8_RECIPE_BLOCKWISE_POW2;
        if (op != FP8_GEMM_FWD && op != FP8_GEMM_DGRAD && op != FP8_GEMM_WGRAD)
            return fail(FP8_ERR_INVALID_ARG, "unknown op %d", op);
        if (d_dtype != FP8_OUT_BF16) return fail(FP8_ERR_UNSUPPORTED, "this recipe's GEMM writes bf16 only");
        s = check_out(A, "A", recipe, FP8_LAYOUT_MX_1x32, M, K);
        if (s != FP8_OK) return s;
        s = check_out(B, "B", recipe, FP8_LAYOUT_MX_1x32, N, K);
        if (s != FP8_OK) return s;
        uint8_t* qc = nullptr;
        uint8_t* qs = nullptr;
        if (d_quant != nullptr) {
            if (N % 128 != 0) return fail(FP8_ERR_UNSUPPORTED, "fused quantization needs N %% 128 == 0");
            s = check_out(d_quant, "d_quant", recipe, FP8_LAYOUT_MX_1x32, M, N);
            if (s != FP8_OK) return s;
            qc = static_cast<uint8_t*>(d_quant->codes);
            qs = static_cast<uint8_t*>(d_quant->scales);
        }
        GemmMxArgs a;
        a.a_codes = static_cast<const uint8_t*>(A->codes);
        a.b_codes = static_cast<const uint8_t*>(B->codes);
        a.sfa = static_cast<const uint8_t*>(A->scales);
        a.sfb = static_cast<const uint8_t*>(B->scales);
        a.M = M;
        a.N = N;
        a.K = K;
        a.m_offsets = nullptr;
        a.G = 1;
        a.D = D;
        a.ldd = ldd;
        a.q_codes = qc;
        a.q_scales = qs;
        a.q_pow2 = pow2;
        cudaError_t e = launch_gemm_mx(a, st, cs);
        return e == cudaSuccess ? FP8_OK : cuda_fail(e, "gemm_blockscaled(mx)");
    }
    return fail(FP8_ERR_INVALID_ARG, "A: unknown recipe %d", A->recipe);
}

fp8_status fp8_grouped_gemm(const fp8_tensor* A, const fp8_tensor* B_stack, const int32_t* m_offsets_dev,
                            int32_t num_groups, int64_t N, void* D, int64_t ldd, fp8_stream_t stream) {
    if (A == nullptr || B_stack == nullptr || m_offsets_dev == nullptr)
        return fail(FP8_ERR_INVALID_ARG, "NULL argument");
    if (num_groups < 1 || num_groups > 1024) return fail(FP8_ERR_UNSUPPORTED, "num_groups must be in [1, 1024]");
    const int64_t total = A->rows, K = A->cols;
    if (N <= 0 || N % 256 != 0) return fail(FP8_ERR_UNSUPPORTED, "grouped GEMM needs N %% 256 == 0 (N = %lld)", (long long)N);
    if (K <= 0 || K % 128 != 0) return fail(FP8_ERR_UNSUPPORTED, "grouped GEMM needs K %% 128 == 0");
    if (total < 0 || total > INT32_MAX / 2) return fail(FP8_ERR_UNSUPPORTED, "bad total rows");
    fp8_status s = check_out(A, "A", FP8_RECIPE_MXFP8, FP8_LAYOUT_MX_1x32_GROUPED, total, K);
    if (s != FP8_OK) return s;
    s = check_out(B_stack, "B_stack", FP8_RECIPE_MXFP8, FP8_LAYOUT_MX_1x32, (int64_t)num_groups * N, K);
    if (s != FP8_OK) return s;
    if (total > 0 && D == nullptr) return fail(FP8_ERR_INVALID_ARG, "D is NULL");
    if (!aligned16(D) || ldd < N || ldd % 8 != 0) return fail(FP8_ERR_ALIGNMENT, "D not 16-byte aligned or bad ldd");
    if (reinterpret_cast<uintptr_t>(m_offsets_dev) & 3u) return fail(FP8_ERR_ALIGNMENT, "m_offsets misaligned");
    fp8_status se;
    StatusBlock* st = status_block(&se);
    if (st == nullptr) return se;
    GemmMxArgs a;
    a.a_codes = static_cast<const uint8_t*>(A->codes);
    a.b_codes = static_cast<const uint8_t*>(B_stack->codes);
    a.sfa = static_cast<const uint8_t*>(A->scales);
    a.sfb = static_cast<const uint8_t*>(B_stack->scales);
    a.M = total;
    a.N = N;
    a.K = K;
    a.m_offsets = m_offsets_dev;
    a.G = num_groups;
    a.D = D;
    a.ldd = ldd;
    a.q_codes = nullptr;
    a.q_scales = nullptr;
    cudaError_t e = launch_gemm_mx(a, st, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "grouped_gemm");
}

fp8_status fp8_sync_payload_size(const fp8_sync_entry* entries, int32_t n, uint64_t* bytes) {
    if (bytes == nullptr) return fail(FP8_ERR_INVALID_ARG, "bytes is NULL");
    std::vector<EntryLayout> lay;
    return sync_layout(entries, n, &lay, bytes);
}

fp8_status fp8_sync_pack(const fp8_sync_entry* entries, int32_t n, void* payload_dev, uint64_t capacity,
                         uint64_t* used_bytes, fp8_stream_t stream) {
    std::vector<EntryLayout> lay;
    uint64_t total = 0;
    fp8_status s = sync_layout(entries, n, &lay, &total);
    if (s != FP8_OK) return s;
    if (payload_dev == nullptr || (reinterpret_cast<uintptr_t>(payload_dev) & 255u))
        return fail(FP8_ERR_ALIGNMENT, "payload must be a 256-byte aligned device pointer");
    if (capacity < total)
        return fail(FP8_ERR_CAPACITY, "payload needs %llu bytes, capacity %llu", (unsigned long long)total,
                    (unsigned long long)capacity);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* pay = static_cast<uint8_t*>(payload_dev);
    std::vector<uint8_t> h = build_table(entries, n, lay, total);
    const unsigned long long tsum = table_checksum(h);   // the segment words are added on the device
    // A header and table that fit a kernel parameter are written by the pack
    // kernel itself (after the checksum field is zeroed), so the call is pure
    // device work: no host staging and nothing that keeps it out of a CUDA
    // graph.  Larger ones are copied from the host.
    static thread_local ExpectTable hdr;
    const ExpectTable* hdr_ptr = nullptr;
    cudaError_t e;
    if (h.size() <= (size_t)kMaxExpectBytes) {
        hdr.bytes = (uint32_t)h.size();
        memcpy(hdr.data, h.data(), h.size());
        hdr_ptr = &hdr;
        e = cudaMemsetAsync(pay + 32, 0, 8, cs);
        if (e != cudaSuccess) return cuda_fail(e, "sync_pack checksum field");
    } else {
        put64(&h[32], tsum);
        e = cudaMemcpyAsync(pay, h.data(), h.size(), cudaMemcpyHostToDevice, cs);
        if (e != cudaSuccess) return cuda_fail(e, "sync_pack header copy");
    }
    // segments: each covers the bytes up to the next segment start
    std::vector<CopySeg> segs;
    for (int32_t i = 0; i < n; ++i) {
        const EntryLayout& L = lay[(size_t)i];
        const uint64_t data_end = L.scale_bytes ? L.scale_off : (i + 1 < n ? lay[(size_t)i + 1].data_off : total);
        segs.push_back(CopySeg{static_cast<const uint8_t*>(entries[i].t.codes), pay + L.data_off, L.data_bytes,
                               data_end - L.data_off, L.data_off / 8});
        if (L.scale_bytes) {
            const uint64_t sc_end = i + 1 < n ? lay[(size_t)i + 1].data_off : total;
            segs.push_back(CopySeg{static_cast<const uint8_t*>(entries[i].t.scales), pay + L.scale_off,
                                   L.scale_bytes, sc_end - L.scale_off, L.scale_off / 8});
        }
    }
    unsigned long long* csum = reinterpret_cast<unsigned long long*>(pay + 32);
    for (size_t b = 0; b < segs.size() || (b == 0 && hdr_ptr != nullptr); b += kMaxCopySegs) {
        const int cnt = (int)std::min<size_t>(kMaxCopySegs, segs.size() - b);
        e = launch_sync_pack(segs.data() + b, cnt, csum, b == 0 ? hdr_ptr : nullptr, tsum, cs);
        if (e != cudaSuccess) return cuda_fail(e, "sync_pack");
    }
    if (used_bytes) *used_bytes = total;
    return FP8_OK;
}

fp8_status fp8_sync_install(const void* payload_dev, uint64_t bytes, const fp8_sync_entry* dst, int32_t n,
                            fp8_stream_t stream) {
    std::vector<EntryLayout> lay;
    uint64_t total = 0;
    fp8_status s = sync_layout(dst, n, &lay, &total);
    if (s != FP8_OK) return s;
    if (payload_dev == nullptr || (reinterpret_cast<uintptr_t>(payload_dev) & 255u))
        return fail(FP8_ERR_ALIGNMENT, "payload must be a 256-byte aligned device pointer");
    if (bytes < total) return fail(FP8_ERR_BAD_PAYLOAD, "payload of %llu bytes, destinations need %llu",
                                   (unsigned long long)bytes, (unsigned long long)total);
    fp8_status se;
    StatusBlock* st = status_block(&se);
    if (st == nullptr) return se;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    InstallOrder order(cs);
    if (order.error() != cudaSuccess) return cuda_fail(order.error(), "sync_install ordering");
    const uint8_t* pay = static_cast<const uint8_t*>(payload_dev);
    std::vector<uint8_t> expect = build_table(dst, n, lay, total);
    std::vector<CopySeg> segs;
    for (int32_t i = 0; i < n; ++i) {
        const EntryLayout& L = lay[(size_t)i];
        segs.push_back(CopySeg{pay + L.data_off, static_cast<uint8_t*>(dst[i].t.codes), L.data_bytes, 0, 0});
        if (L.scale_bytes)
            segs.push_back(CopySeg{pay + L.scale_off, static_cast<uint8_t*>(dst[i].t.scales), L.scale_bytes, 0, 0});
    }
    cudaError_t e;
    const ExpectTable* et_ptr = nullptr;
    unsigned long long tsum = 0;
    if (expect.size() <= (size_t)kMaxExpectBytes) {
        // every byte of header and table except the checksum must match what
        // the destinations imply: checked on the device by the verify kernel
        // (no host round trip); a mismatch installs nothing and is reported
        // by fp8_status_poll
        static thread_local ExpectTable et;
        et.bytes = (uint32_t)expect.size();
        memcpy(et.data, expect.data(), expect.size());
        et_ptr = &et;
        tsum = table_checksum(expect);
    } else {
        std::vector<uint8_t> got(expect.size());
        e = cudaMemcpyAsync(got.data(), pay, got.size(), cudaMemcpyDeviceToHost, cs);
        if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
        if (e != cudaSuccess) return cuda_fail(e, "sync_install header read");
        if (get64(&got[0]) != kSyncMagic || get32(&got[8]) != kSyncVersion)
            return fail(FP8_ERR_BAD_PAYLOAD, "not a version-2 FP8 sync payload");
        if (get32(&got[12]) != (uint32_t)n)
            return fail(FP8_ERR_BAD_PAYLOAD, "payload has %u entries, %d destinations", get32(&got[12]), n);
        for (size_t i = 0; i < expect.size(); ++i) {
            if (i >= 32 && i < 40) continue;
            if (got[i] != expect[i]) {
                const long long ent = i < kHeaderBytes ? -1 : (long long)((i - kHeaderBytes) / kEntryBytes);
                return fail(FP8_ERR_BAD_PAYLOAD, "payload header/table byte %zu differs (entry %lld)", i, ent);
            }
        }
        put64(&got[32], 0);
        tsum = table_checksum(got);
    }
    // one cooperative kernel (verify, grid barrier, copy) when the device
    // runs it and the segments fit one table; otherwise verify, then copy
    e = launch_sync_install(pay, expect.size(), total, tsum, st, et_ptr, segs.data(), (int)segs.size(), cs);
    if (e == cudaSuccess) return FP8_OK;
    if (e != cudaErrorNotSupported && e != cudaErrorCooperativeLaunchTooLarge) return cuda_fail(e, "sync_install");
    (void)cudaGetLastError();
    e = launch_sync_verify(pay, expect.size(), total, tsum, st, cs, et_ptr);
    if (e != cudaSuccess) return cuda_fail(e, "sync_install verify");
    for (size_t b = 0; b < segs.size(); b += kMaxCopySegs) {
        const int cnt = (int)std::min<size_t>(kMaxCopySegs, segs.size() - b);
        e = launch_sync_scatter(&segs[b], cnt, st, cs);
        if (e != cudaSuccess) return cuda_fail(e, "sync_install scatter");
    }
    return FP8_OK;
}

fp8_status fp8_check_wait_expiry(int64_t limit_ns, fp8_stream_t stream) {
    if (limit_ns < 1000 || limit_ns > 2000000000) return fail(FP8_ERR_INVALID_ARG, "limit_ns must be in [1 us, 2 s]");
    fp8_status se;
    StatusBlock* st = status_block(&se);
    if (st == nullptr) return se;
    cudaError_t e = launch_wait_expiry((unsigned long long)limit_ns, st, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : cuda_fail(e, "check_wait_expiry");
}

fp8_status fp8_status_poll(fp8_stream_t stream) {
    fp8_status se;
    StatusBlock* st = status_block(&se);
    if (st == nullptr) return se;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "status_poll sync");
    unsigned int bits[2] = {0, 0};
    e = cudaMemcpy(bits, st, sizeof(bits), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status_poll read");
    if (bits[0] == 0) return FP8_OK;
    e = cudaMemset(st, 0, 2 * sizeof(unsigned int));
    if (e != cudaSuccess) return cuda_fail(e, "status_poll clear");
    if (bits[0] & kErrTimeout)
        return fail(FP8_ERR_TIMEOUT, "a bounded on-chip wait expired (site %u)", bits[1]);
    if (bits[0] & kErrBadPayload)
        return fail(FP8_ERR_BAD_PAYLOAD, "sync payload header/table does not match the destinations; nothing installed");
    if (bits[0] & kErrChecksum) return fail(FP8_ERR_CHECKSUM, "sync payload checksum mismatch; nothing installed");
    return fail(FP8_ERR_INVALID_ARG, "a kernel rejected a device-side argument (e.g. a gather index)");
}

// Install for callers that cannot allocate device memory; see fp8bs.h.
fp8_status fp8_sync_install_noalloc(const void* payload_dev, uint64_t bytes, const fp8_sync_entry* dst, int32_t n,
                                    fp8_stream_t stream) {
    if (n < 0 || (n > 0 && dst == nullptr)) return fail(FP8_ERR_INVALID_ARG, "bad entry list");
    if (n > kNoAllocMaxEntries)
        return fail(FP8_ERR_CAPACITY, "fp8_sync_install_noalloc takes at most %d entries (got %d); "
                    "use fp8_sync_install", kNoAllocMaxEntries, n);
    if (payload_dev == nullptr || (reinterpret_cast<uintptr_t>(payload_dev) & 255u))
        return fail(FP8_ERR_ALIGNMENT, "payload must be a 256-byte aligned device pointer");
    EntryLayout lay[kNoAllocMaxEntries];
    uint64_t off = round_up(kHeaderBytes + kEntryBytes * (uint64_t)n, 256);
    const uint64_t data_offset = off;
    for (int32_t i = 0; i < n; ++i) {
        uint64_t db, sb;
        fp8_status s = entry_bytes(dst[i], i, &db, &sb);
        if (s != FP8_OK) return s;
        lay[i].data_off = off;
        lay[i].data_bytes = db;
        off = round_up(off + db, 256);
        lay[i].scale_off = sb ? off : 0;
        lay[i].scale_bytes = sb;
        off = round_up(off + sb, 256);
    }
    const uint64_t total = off;
    if (bytes < total)
        return fail(FP8_ERR_BAD_PAYLOAD, "payload of %llu bytes, destinations need %llu", (unsigned long long)bytes,
                    (unsigned long long)total);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    InstallOrder order(cs);
    if (order.error() != cudaSuccess) return cuda_fail(order.error(), "sync_install_noalloc ordering");
    const uint8_t* pay = static_cast<const uint8_t*>(payload_dev);

    // header and table: read back and compare with what dst implies
    uint8_t expect[kNoAllocTableBytes];
    uint8_t got[kNoAllocTableBytes];
    fill_table(expect, data_offset, dst, n, lay, total);
    cudaError_t e = cudaMemcpyAsync(got, pay, (size_t)data_offset, cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "sync_install_noalloc header read");
    if (get64(&got[0]) != kSyncMagic || get32(&got[8]) != kSyncVersion)
        return fail(FP8_ERR_BAD_PAYLOAD, "not a version-2 FP8 sync payload");
    if (get32(&got[12]) != (uint32_t)n)
        return fail(FP8_ERR_BAD_PAYLOAD, "payload has %u entries, %d destinations", get32(&got[12]), n);
    for (uint64_t i = 0; i < data_offset; ++i) {
        if (i >= 32 && i < 40) continue;
        if (got[i] != expect[i]) return fail(FP8_ERR_BAD_PAYLOAD, "payload header/table byte %llu differs",
                                             (unsigned long long)i);
    }
    put64(&got[32], 0);
    unsigned long long table_sum = 0;
    for (uint64_t i = kHeaderBytes / 8; i < data_offset / 8; ++i) table_sum += word_term(get64(&got[8 * i]), i);

    fp8_status se;
    NoAllocScratch* sc = noalloc_scratch(&se);
    if (sc == nullptr) return se;
    CopySeg segs[kNoAllocMaxSegs];
    int nseg = 0;
    for (int32_t i = 0; i < n; ++i) {
        segs[nseg++] = CopySeg{pay + lay[i].data_off, static_cast<uint8_t*>(dst[i].t.codes), lay[i].data_bytes, 0, 0};
        if (lay[i].scale_bytes)
            segs[nseg++] =
                CopySeg{pay + lay[i].scale_off, static_cast<uint8_t*>(dst[i].t.scales), lay[i].scale_bytes, 0, 0};
    }
    // the previous call's contents stay in the array: clear the status part
    e = cudaMemsetAsync(&sc->status, 0, sizeof(StatusBlock), cs);
    if (e == cudaSuccess && nseg > 0)
        e = cudaMemcpyAsync(sc->segs, segs, sizeof(CopySeg) * (size_t)nseg, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return cuda_fail(e, "sync_install_noalloc set-up");
    e = launch_sync_verify(pay, data_offset, total, table_sum, &sc->status, cs);
    if (e != cudaSuccess) return cuda_fail(e, "sync_install_noalloc verify");
    if (nseg > 0) {
        // grid: the 256-thread blocks the copy needs, capped by what is
        // resident on this device at once (SM count x blocks per SM)
        uint64_t chunks = 0;
        for (int i = 0; i < nseg; ++i) chunks += (segs[i].bytes + 15) / 16;
        static int resident[64] = {};
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e, "sync_install_noalloc device");
        int& r = resident[dev & 63];
        if (r == 0) {
            int sms = 0, per_sm = 0;
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_sync_scatter_table, 256, 0);
            r = (sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
        }
        const uint64_t need = (chunks + 255) / 256;
        const unsigned grid = (unsigned)(need < 1 ? 1 : (need < (uint64_t)r ? need : (uint64_t)r));
        k_sync_scatter_table<<<grid, 256, 0, cs>>>(sc, nseg);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "sync_install_noalloc scatter");
    }
    unsigned int verdict = 1;
    e = cudaMemcpyAsync(&verdict, &sc->status.verdict, sizeof(verdict), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "sync_install_noalloc verdict read");
    if (verdict != 0) return fail(FP8_ERR_CHECKSUM, "sync payload checksum mismatch; nothing installed");
    return FP8_OK;
}

}  // extern "C"
