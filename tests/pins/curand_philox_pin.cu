// Test-only pin for the oracle's Philox4x32-10: exposes, as a host function,
// the curand library's own Philox4x32-10 block function (curand_philox4x32_x.h
// from the CUDA toolkit), compiled for the host. The header lets the caller
// choose the function qualifiers; nothing of it is copied here, it is called.
#define QUALIFIERS static inline __host__ __device__
#include <curand_philox4x32_x.h>

extern "C" void pin_curand_philox4x32_10(const unsigned int* ctr, const unsigned int* key,
                                         unsigned int* out, int n) {
  for (int i = 0; i < n; ++i) {
    uint4 c = make_uint4(ctr[4 * i + 0], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
    uint2 k = make_uint2(key[2 * i + 0], key[2 * i + 1]);
    uint4 r = curand_Philox4x32_10(c, k);
    out[4 * i + 0] = r.x;
    out[4 * i + 1] = r.y;
    out[4 * i + 2] = r.z;
    out[4 * i + 3] = r.w;
  }
}
