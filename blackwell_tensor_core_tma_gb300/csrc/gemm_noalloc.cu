// gemm_run_noalloc: the bf16/fp16 GEMM for callers that cannot allocate
// device memory (see include/gb300gemm.h).
//
// The only global memory the kernel uses beyond its inputs and outputs is its
// status word.  The plan API allocates that word with cudaMalloc; here it
// lives in a file-scope __device__ array instead, so a call allocates
// nothing.  In host code `g_noalloc_scratch` is only a host-side stand-in for
// the symbol: its device address comes from cudaGetSymbolAddress, taken once
// per device (with that device current) on the first call there.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "gemm_internal.h"
#include "ptx.cuh"

using namespace gb300;

namespace {

constexpr size_t kScratchBytes = 256;                  // capacity of the array
constexpr size_t kStatusBytes = sizeof(int);           // what the kernel needs: its status word
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceState {
    bool ready;
    int *status;          // device address of g_noalloc_scratch on this device
    int sm_count;
    int pair_clusters;    // co-resident CTA pairs of the cta_group::2 kernel
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;

gemm_status setup(int dev, DeviceState **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return GEMM_ERR_CUDA;
        if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_UNSUPPORTED;
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return GEMM_ERR_CUDA;
        for (int cg = 1; cg <= 2; ++cg)
            for (int bf = 0; bf <= 1; ++bf)
                if (f16_prepare(F16Config{cg, bf}) != cudaSuccess) return GEMM_ERR_CUDA;
        int clusters = 0;
        if (f16_max_active_clusters(F16Config{2, 1}, &clusters) != cudaSuccess || clusters <= 0)
            clusters = prop.multiProcessorCount / 2;
        if (!g_enc) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess)
                return GEMM_ERR_CUDA;
            g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        s.status = static_cast<int *>(ptr);
        s.sm_count = prop.multiProcessorCount;
        s.pair_clusters = clusters;
        s.ready = true;
    }
    *out = &s;
    return GEMM_OK;
}

bool encode(CUtensorMap *m, CUtensorMapDataType dt, int ebytes, const void *ptr, uint64_t inner, uint64_t outer,
            uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (uint64_t)ebytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_enc(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" gemm_status gemm_run_noalloc(int64_t M, int64_t N, int64_t K, gemm_dtype ab, gemm_dtype d,
                                        const void *A, const void *B, const void *C, void *D, void *cuda_stream,
                                        int wait) {
    if (M <= 0 || N <= 0 || K <= 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if (!A || !B || !D) return GEMM_ERR_INVALID_ARG;
    if (kStatusBytes > kScratchBytes) return GEMM_ERR_INVALID_ARG;   // scratch beyond the array's capacity
    if (ab != GEMM_F16 && ab != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
    if (d != GEMM_F32 && d != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
    const int dbytes = d == GEMM_BF16 ? 2 : 4;
    if ((K * 2) % 16 != 0 || (N * 4) % 16 != 0 || (N * dbytes) % 16 != 0) return GEMM_ERR_ALIGNMENT;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (C && !aligned16(C))) return GEMM_ERR_ALIGNMENT;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    DeviceState *s = nullptr;
    gemm_status st = setup(dev, &s);
    if (st != GEMM_OK) return st;

    // the CTA mode a plan without flags would choose, but always 128 x 256 (single CTA) or
    // 256 x 256 (pair) tiles, the 4-warp epilogue, groups of 8 pair tiles (16 single-CTA
    // tiles) and no split-K or stream-K: a plan may pick other forms of the kernel
    const int cg = (M >= 1024 && N >= 1024) ? 2 : 1;
    const F16Config cfg{cg, d == GEMM_BF16};
    CUtensorMap maps[NUM_MAPS];
    std::memset(maps, 0, sizeof maps);
    const CUtensorMapDataType abt = ab == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    bool ok = encode(&maps[0], abt, 2, A, K, M, TILE_K16, TILE_M, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode(&maps[1], abt, 2, B, K, N, TILE_K16, TILE_N / cg, CU_TENSOR_MAP_SWIZZLE_128B);
    if (ok && C)
        ok = encode(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, N, M, EPI_COLS, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (ok)
        ok = d == GEMM_BF16
                 ? encode(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, N, M, EPI_COLS, 32, CU_TENSOR_MAP_SWIZZLE_64B)
                 : encode(&maps[3], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, N, M, EPI_COLS, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return GEMM_ERR_CUDA;

    KParams kp{};
    kp.M = (int)M;
    kp.N = (int)N;
    kp.K = (int)K;
    kp.tiles_m = (int)((M + TILE_M * cg - 1) / (TILE_M * cg));
    kp.tiles_n = (int)((N + TILE_N - 1) / TILE_N);
    kp.num_tiles = kp.tiles_m * kp.tiles_n;
    kp.num_kb = (int)((K + TILE_K16 - 1) / TILE_K16);
    kp.group_m = cg == 2 ? 8 : 16;
    kp.has_c = C != nullptr;
    kp.splits = 1;
    kp.idesc = idesc_f16(ab == GEMM_BF16 ? 1u : 0u, (uint32_t)(TILE_M * cg), (uint32_t)TILE_N);
    kp.status = s->status;
    kp.timeout_ns = 1000000000ull;
    kp.fault = 0;
    const int units = cg == 2 ? s->pair_clusters : s->sm_count;
    LaunchShape shape{cg * (kp.num_tiles < units ? kp.num_tiles : units), cg, f16_smem_bytes(cfg)};

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    if (wait) {
        // waiting would synchronise a stream that is being captured into a graph, which
        // fails and invalidates the capture: refuse before enqueueing anything
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return GEMM_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return GEMM_ERR_INVALID_ARG;
    }
    // the array keeps the previous call's status: it must start at zero
    if (cudaMemsetAsync(s->status, 0, kStatusBytes, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    if (f16_launch(cfg, shape, maps, kp, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    if (!wait) return GEMM_OK;
    int v = 0;
    if (cudaMemcpyAsync(&v, s->status, kStatusBytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return (gemm_status)v;
}
