// w4_api.cu -- the extern "C" boundary (declared in include/w4.h).
//
// Every entry point validates its arguments on the host, before anything is
// enqueued, and then launches its kernel(s) on the caller's stream.  No entry
// point allocates, synchronises or keeps state between calls.

#include "common.cuh"

namespace w4 {

w4_status run_quantize_pack(const void* W, void* packed, float* scale, int64_t K, int64_t N, cudaStream_t s);
w4_status run_permute(const void* packed, void* out, int64_t K, int64_t N, cudaStream_t s);
w4_status run_quantize_pack_permute(const void* W, void* out, float* scale, int64_t K, int64_t N, cudaStream_t s);
w4_status run_gemv(const void* qw, const void* scale, const void* zero, const void* x, void* d, int64_t N,
                   int64_t K, int64_t C, w4_dtype dtype, cudaStream_t s);
w4_status run_gemm(const void* A, const void* B, const void* scale, const void* zero, void* C, int64_t M,
                   int64_t N, int64_t K, cudaStream_t s);
w4_status run_gemv_permuted(const void* permuted, const float* scale, const void* x, void* d, int N, int K, int C,
                            cudaStream_t s);
w4_status run_quantize_int8(const void* W, void* q, float* scale, int64_t K, int64_t N, cudaStream_t s);
w4_status run_permute_int8(const void* q, void* out, int64_t K, int64_t N, cudaStream_t s);
w4_status run_gemv_w8(const void* q, const float* scale, const void* x, void* d, int64_t N, int64_t K, int64_t C,
                      cudaStream_t s);
w4_status run_quantize_q8_1_pt(const void* x, void* pt, int64_t C, int64_t K, cudaStream_t s);
w4_status run_gemv_w4a8(const void* qw, const void* scale, const void* zero, const void* pt, void* d, int64_t N,
                        int64_t K, int64_t C, cudaStream_t s);
bool w4a8_fits(int64_t C, int64_t K);
w4_status run_mmvq_ptq1_0(const void* blocks, const void* pt, float* d, int64_t N, int64_t K, int64_t C,
                          cudaStream_t s);
w4_status run_mmvq_ptq1_1(const void* sblocks, const void* codebook, int64_t n_code, const void* esc_idx,
                          const void* esc_patt, int64_t n_esc, const void* pt, float* d, int64_t N, int64_t K,
                          int64_t C, cudaStream_t s);
bool ptq1_fits(int64_t C, int64_t K, bool super);
int take_device_error_ptq1();
w4_status run_selftest_wait_timeout(int* waited, cudaStream_t s);
int take_device_error_selftest();
w4_status run_gemm_w8(const void* A, const void* q, const float* scale, void* C, int64_t M, int64_t N, int64_t K,
                      cudaStream_t s);
w4_status run_gemm_w4_permuted(const void* A, const void* permuted, const float* scale, void* C, int64_t M,
                               int64_t N, int64_t K, cudaStream_t s);
int take_device_error_gemm();
int take_device_error_gemv();
int take_device_error_quant();
int set_wait_limit_gemm(long long clocks);
int set_wait_limit_gemv(long long clocks);
int set_wait_limit_quant(long long clocks);
int set_wait_limit_ptq1(long long clocks);
int set_wait_limit_selftest(long long clocks);
int set_short_first_stage_gemv(int on);
int set_short_first_stage_gemm(int on);

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
int g_is_sm103[kMaxDevices];  // 0 unknown, 1 yes, -1 no
}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

bool device_is_sm103() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (g_is_sm103[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return false;
        g_is_sm103[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_is_sm103[dev] == 1;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace w4

using namespace w4;

extern "C" {

int w4_abi_version(void) { return 4; }

int w4_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
    const int a = take_device_error_gemm();
    const int b = take_device_error_gemv();
    const int c = take_device_error_quant();
    const int e = take_device_error_ptq1();
    const int f = take_device_error_selftest();
    if (a < 0 || b < 0 || c < 0 || e < 0 || f < 0) return -1;
    return a != 0 ? a : b != 0 ? b : c != 0 ? c : e != 0 ? e : f;
}

const char* w4_status_string(w4_status status) {
    switch (status) {
        case W4_OK: return "ok";
        case W4_ERR_NULL: return "null pointer argument";
        case W4_ERR_SHAPE: return "illegal size or shape";
        case W4_ERR_ALIGN: return "pointer not 16-byte aligned";
        case W4_ERR_DTYPE: return "unsupported dtype";
        case W4_ERR_CUDA: return "CUDA launch error";
        case W4_ERR_DEVICE: return "current device is not an sm_103 (GB300) GPU";
        case W4_ERR_VALUE: return "input value outside the format's range";
    }
    return "unknown status";
}

w4_status quantize_pack_int4(const void* W, void* packed, float* scale, int64_t K, int64_t N, void* stream) {
    if (K < 0 || N < 0 || (K % 2) != 0) return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!scale || (K > 0 && (!W || !packed))) return W4_ERR_NULL;
    if (!aligned16(scale) || (K > 0 && (!aligned16(W) || !aligned16(packed)))) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(scale, 0, N * sizeof(float), (cudaStream_t)stream));
    return run_quantize_pack(W, packed, scale, K, N, (cudaStream_t)stream);
}

w4_status quantize_pack_permute_int4(const void* W, void* permuted, float* scale, int64_t K, int64_t N,
                                     void* stream) {
    if (K < 0 || N < 0 || (K % 64) != 0 || (N % 8) != 0 || K > W4_QUANT_PERMUTE_MAX_K) return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!scale || (K > 0 && (!W || !permuted))) return W4_ERR_NULL;
    if (!aligned16(scale) || (K > 0 && (!aligned16(W) || !aligned16(permuted)))) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(scale, 0, N * sizeof(float), (cudaStream_t)stream));
    return run_quantize_pack_permute(W, permuted, scale, K, N, (cudaStream_t)stream);
}

w4_status permute_int4(const void* packed, void* out, int64_t K, int64_t N, void* stream) {
    if (K < 0 || N < 0 || (K % 64) != 0 || (N % 4) != 0) return W4_ERR_SHAPE;
    if (K == 0 || N == 0) return W4_OK;
    if (!packed || !out) return W4_ERR_NULL;
    if (!aligned16(packed) || !aligned16(out)) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    return run_permute(packed, out, K, N, (cudaStream_t)stream);
}

w4_status gemv_w4(const void* qweight, const void* scale, const void* zero, const void* x, void* d, int64_t N,
                  int64_t K, int64_t C, w4_dtype dtype, void* stream) {
    if (dtype != W4_F32 && dtype != W4_BF16) return W4_ERR_DTYPE;
    if (N < 0 || K < 0 || (K % 8) != 0 || K > W4_GEMV_MAX_K || C < 1 || C > 8) return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!d || !scale || !zero || (K > 0 && (!qweight || !x))) return W4_ERR_NULL;
    if (!aligned16(d) || !aligned16(scale) || !aligned16(zero) ||
        (K > 0 && (!aligned16(qweight) || !aligned16(x))))
        return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    const size_t esz = dtype == W4_F32 ? 4 : 2;
    if (K == 0) return launch_status(cudaMemsetAsync(d, 0, C * N * esz, (cudaStream_t)stream));
    return run_gemv(qweight, scale, zero, x, d, N, K, C, dtype, (cudaStream_t)stream);
}

w4_status gemv_w4_permuted(const void* permuted, const float* scale, const void* x, void* d, int64_t N, int64_t K,
                          int64_t C, void* stream) {
    if (N < 0 || K < 0 || (K % 64) != 0 || (N % 4) != 0 || K > W4_GEMV_MAX_K || C < 1 || C > 8 ||
        N > (int64_t(1) << 30))
        return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!d || !scale || (K > 0 && (!permuted || !x))) return W4_ERR_NULL;
    if (!aligned16(d) || !aligned16(scale) || (K > 0 && (!aligned16(permuted) || !aligned16(x)))) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(d, 0, C * N * 2, (cudaStream_t)stream));
    return run_gemv_permuted(permuted, scale, x, d, static_cast<int>(N), static_cast<int>(K), static_cast<int>(C),
                             (cudaStream_t)stream);
}

w4_status quantize_int8(const void* W, void* q, float* scale, int64_t K, int64_t N, void* stream) {
    if (K < 0 || N < 0) return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!scale || (K > 0 && (!W || !q))) return W4_ERR_NULL;
    if (!aligned16(scale) || (K > 0 && (!aligned16(W) || !aligned16(q)))) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(scale, 0, N * sizeof(float), (cudaStream_t)stream));
    return run_quantize_int8(W, q, scale, K, N, (cudaStream_t)stream);
}

w4_status permute_int8(const void* q, void* out, int64_t K, int64_t N, void* stream) {
    if (K < 0 || N < 0 || (K % 64) != 0 || (N % 2) != 0) return W4_ERR_SHAPE;
    if (K == 0 || N == 0) return W4_OK;
    if (!q || !out) return W4_ERR_NULL;
    if (!aligned16(q) || !aligned16(out)) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    return run_permute_int8(q, out, K, N, (cudaStream_t)stream);
}

w4_status gemv_w8(const void* q, const float* scale, const void* x, void* d, int64_t N, int64_t K, int64_t C,
                  void* stream) {
    if (N < 0 || K < 0 || C < 1 || C > 8) return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!d || !scale || (K > 0 && (!q || !x))) return W4_ERR_NULL;
    if (!aligned16(d) || !aligned16(scale) || (K > 0 && (!aligned16(q) || !aligned16(x)))) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(d, 0, C * N * 2, (cudaStream_t)stream));
    return run_gemv_w8(q, scale, x, d, N, K, C, (cudaStream_t)stream);
}

w4_status quantize_q8_1_pt(const void* x, void* pt, int64_t C, int64_t K, void* stream) {
    if (C < 0 || K < 0 || (K % 128) != 0) return W4_ERR_SHAPE;
    if (C == 0 || K == 0) return W4_OK;
    if (!x || !pt) return W4_ERR_NULL;
    if (!aligned16(x) || !aligned16(pt)) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    return run_quantize_q8_1_pt(x, pt, C, K, (cudaStream_t)stream);
}

w4_status gemv_w4a8(const void* qweight, const void* scale, const void* zero, const void* pt, void* d, int64_t N,
                    int64_t K, int64_t C, void* stream) {
    if (N < 0 || K < 0 || (K % 128) != 0 || C < 1 || C > 8 || !w4a8_fits(C, K)) return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!d || !scale || !zero || (K > 0 && (!qweight || !pt))) return W4_ERR_NULL;
    if (!aligned16(d) || !aligned16(scale) || !aligned16(zero) || (K > 0 && (!aligned16(qweight) || !aligned16(pt))))
        return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(d, 0, C * N * 2, (cudaStream_t)stream));
    return run_gemv_w4a8(qweight, scale, zero, pt, d, N, K, C, (cudaStream_t)stream);
}

w4_status mmvq_ptq1_0(const void* blocks, const void* pt, float* d, int64_t N, int64_t K, int64_t C, void* stream) {
    if (N < 0 || K < 0 || (K % 128) != 0 || C < 1 || C > 8 || !ptq1_fits(C, K, false)) return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!d || (K > 0 && (!blocks || !pt))) return W4_ERR_NULL;
    if (!aligned16(d) || (K > 0 && (!aligned16(blocks) || !aligned16(pt)))) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(d, 0, C * N * sizeof(float), (cudaStream_t)stream));
    return run_mmvq_ptq1_0(blocks, pt, d, N, K, C, (cudaStream_t)stream);
}

w4_status mmvq_ptq1_1(const void* sblocks, const void* codebook, int64_t n_code, const void* esc_idx,
                      const void* esc_patt, int64_t n_esc, const void* pt, float* d, int64_t N, int64_t K, int64_t C,
                      void* stream) {
    if (N < 0 || K < 0 || (K % 128) != 0 || C < 1 || C > 8 || n_code < 0 || n_code > 767 || n_esc < 0 ||
        !ptq1_fits(C, K, true))
        return W4_ERR_SHAPE;
    if (N == 0) return W4_OK;
    if (!d || (K > 0 && (!sblocks || !pt)) || (n_code > 0 && !codebook) || (n_esc > 0 && (!esc_idx || !esc_patt)))
        return W4_ERR_NULL;
    if (!aligned16(d) || (K > 0 && (!aligned16(sblocks) || !aligned16(pt))) || (n_code > 0 && !aligned16(codebook)) ||
        (n_esc > 0 && (!aligned16(esc_idx) || !aligned16(esc_patt))))
        return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(d, 0, C * N * sizeof(float), (cudaStream_t)stream));
    return run_mmvq_ptq1_1(sblocks, codebook, n_code, esc_idx, esc_patt, n_esc, pt, d, N, K, C, (cudaStream_t)stream);
}

w4_status gemm_w8(const void* A, const void* q, const float* scale, void* C, int64_t M, int64_t N, int64_t K,
                  void* stream) {
    if (M < 0 || N < 0 || K < 0 || (K % 64) != 0 || (N % 16) != 0) return W4_ERR_SHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!C || !scale || (K > 0 && (!A || !q))) return W4_ERR_NULL;
    if (!aligned16(C) || !aligned16(scale) || (K > 0 && (!aligned16(A) || !aligned16(q)))) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(C, 0, M * N * 2, (cudaStream_t)stream));
    return run_gemm_w8(A, q, scale, C, M, N, K, (cudaStream_t)stream);
}

w4_status gemm_w4_permuted(const void* A, const void* permuted, const float* scale, void* C, int64_t M, int64_t N,
                           int64_t K, void* stream) {
    if (M < 0 || N < 0 || K < 0 || (K % 64) != 0 || (N % 16) != 0) return W4_ERR_SHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!C || !scale || (K > 0 && (!A || !permuted))) return W4_ERR_NULL;
    if (!aligned16(C) || !aligned16(scale) || (K > 0 && (!aligned16(A) || !aligned16(permuted)))) return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(C, 0, M * N * 2, (cudaStream_t)stream));
    return run_gemm_w4_permuted(A, permuted, scale, C, M, N, K, (cudaStream_t)stream);
}

w4_status w4_selftest_configure(long long wait_limit_clocks, int short_first_stage) {
    const long long limit = wait_limit_clocks > 0 ? wait_limit_clocks : (1ll << 32);
    if (cudaDeviceSynchronize() != cudaSuccess) return W4_ERR_CUDA;
    if (set_wait_limit_gemm(limit) || set_wait_limit_gemv(limit) || set_wait_limit_quant(limit) ||
        set_wait_limit_ptq1(limit) || set_wait_limit_selftest(limit) ||
        set_short_first_stage_gemv(short_first_stage) || set_short_first_stage_gemm(short_first_stage))
        return W4_ERR_CUDA;
    return W4_OK;
}

w4_status w4_selftest_wait_timeout(int* waited, void* stream) {
    if (!waited) return W4_ERR_NULL;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    return run_selftest_wait_timeout(waited, (cudaStream_t)stream);
}

w4_status gemm_w4(const void* A, const void* B, const void* scale, const void* zero, void* C, int64_t M, int64_t N,
                  int64_t K, void* stream) {
    if (M < 0 || N < 0 || K < 0 || (K % 64) != 0 || (N % 16) != 0) return W4_ERR_SHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!C || !scale || !zero || (K > 0 && (!A || !B))) return W4_ERR_NULL;
    if (!aligned16(C) || !aligned16(scale) || !aligned16(zero) || (K > 0 && (!aligned16(A) || !aligned16(B))))
        return W4_ERR_ALIGN;
    if (!device_is_sm103()) return W4_ERR_DEVICE;
    if (K == 0) return launch_status(cudaMemsetAsync(C, 0, M * N * 2, (cudaStream_t)stream));
    return run_gemm(A, B, scale, zero, C, M, N, K, (cudaStream_t)stream);
}

}  // extern "C"
