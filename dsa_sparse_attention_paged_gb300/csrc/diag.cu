// diag.cu -- diagnostic kernels that run the library's own device functions
// on caller-chosen inputs: the coarse bin over a range of FP32 bit patterns,
// the packed FP16 order-key transform, and a bounded wait that is made to run
// out (to show that a wait records DSA_DEV_TIMEOUT and returns).
#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {

namespace {

__global__ void bins_range_kernel(uint32_t start, int64_t count, int16_t *out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t u = start + (uint32_t)i;
    out[i] = (int16_t)coarse_bin(__uint_as_float(u));
  }
}

__global__ void fp16_keys_kernel(const uint32_t *in, uint32_t *out, int64_t nw) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nw;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = f16x2_order_keys(in[i]);
}

__global__ void bf16_keys_kernel(const uint32_t *in, uint32_t *out, int64_t nw) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nw;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = bf16x2_order_keys(in[i]);
}

// One thread waits on a barrier that expects one arrival nobody makes.
__global__ void wait_selftest_kernel(long long limit, uint32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl ctl{&abort_flag, status, limit};
    (void)mbar_wait(smem_u32(&bar), 0, ctl);
  }
}

}  // namespace

dsa_status_t run_bins_range(uint32_t start, int64_t count, int16_t *out, cudaStream_t st) {
  if (count <= 0) return DSA_OK;
  const int sms = num_sms();
  if (sms <= 0) return DSA_ERR_CUDA;
  bins_range_kernel<<<sms * 8, 256, 0, st>>>(start, count, out);
  return check_launch();
}

dsa_status_t run_fp16_keys(const uint16_t *in, uint16_t *out, int64_t n, cudaStream_t st) {
  if (n <= 0) return DSA_OK;
  const int sms = num_sms();
  if (sms <= 0) return DSA_ERR_CUDA;
  fp16_keys_kernel<<<sms * 4, 256, 0, st>>>(reinterpret_cast<const uint32_t *>(in),
                                             reinterpret_cast<uint32_t *>(out), n / 2);
  return check_launch();
}

dsa_status_t run_bf16_keys(const uint16_t *in, uint16_t *out, int64_t n, cudaStream_t st) {
  if (n <= 0) return DSA_OK;
  const int sms = num_sms();
  if (sms <= 0) return DSA_ERR_CUDA;
  bf16_keys_kernel<<<sms * 4, 256, 0, st>>>(reinterpret_cast<const uint32_t *>(in),
                                             reinterpret_cast<uint32_t *>(out), n / 2);
  return check_launch();
}

dsa_status_t run_wait_selftest(uint64_t limit, uint32_t *status, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>((long long)limit, status);
  return check_launch();
}

}  // namespace dsa
