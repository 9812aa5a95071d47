// One-time weight preparation: the fp16 copy of a down-projection matrix
// that the tensor-core prefill path multiplies h by (h is kept in fp16 for
// its 11-bit significand; both MMA operands of one UMMA must share a type).
// The conversion is exact for |w| >= 2^-14 (smaller magnitudes become fp16
// subnormals, absolute error <= 2^-25); |w| >= 65520 has no fp16 value and
// is recorded as MM_ERR_RANGE in the status header.
#include "mm_kernels.cuh"

namespace mm {

__global__ void prepare_wd16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                    int64_t nvec, WsHeader* hdr) {
  bool bad = false;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 r = src[i];
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a = __uint_as_float(w[q] << 16), b = __uint_as_float(w[q] & 0xffff0000u);
      bad |= !(fabsf(a) < 65520.0f) | !(fabsf(b) < 65520.0f);
      o[q] = pack_f16x2(a, b);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && hdr != nullptr)
    if (atomicCAS(&hdr->status, 0u, kStatusRange) == 0u) hdr->where = 101;
}

cudaError_t launch_prepare_wd16(const void* Wd, void* Wd16, int64_t n, WsHeader* hdr,
                                cudaStream_t st) {
  const int64_t nvec = n / 8;
  const int64_t want = (nvec + 255) / 256;
  const int grid = static_cast<int>(want < 4L * num_sms() ? (want > 0 ? want : 1) : 4L * num_sms());
  prepare_wd16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(Wd), static_cast<uint4*>(Wd16),
                                            nvec, hdr);
  return cudaGetLastError();
}

}  // namespace mm
