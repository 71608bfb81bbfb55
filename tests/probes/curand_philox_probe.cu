// Test-only probe: evaluates cuRAND's device Philox4x32-10 (curand_kernel.h)
// on caller-given counters and keys, so the tests can compare the oracle's
// Philox with an implementation written by others.  Not part of the library.
#include <curand_kernel.h>
#include <stdint.h>

__global__ void philox_probe_kernel(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint4 c = make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
    const uint2 k = make_uint2(key[2 * i], key[2 * i + 1]);
    const uint4 r = curand_Philox4x32_10(c, k);
    out[4 * i] = r.x;
    out[4 * i + 1] = r.y;
    out[4 * i + 2] = r.z;
    out[4 * i + 3] = r.w;
}

// d_ctr: n x 4 words, d_key: n x 2 words, d_out: n x 4 words (device).
extern "C" int philox_probe(const uint32_t* d_ctr, const uint32_t* d_key, uint32_t* d_out, int n)
{
    if (n <= 0) return 0;
    philox_probe_kernel<<<(n + 255) / 256, 256>>>(d_ctr, d_key, d_out, n);
    return (int)cudaDeviceSynchronize();
}
