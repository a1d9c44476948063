// curand_philox.cu -- test infrastructure: prints the output block of cuRAND's
// Philox4_32_10 generator for (seed, subsequence, counter) triples read from
// stdin, one "x y z w" line (hex) per triple.  With offset 4 * counter,
// curand_init leaves the generator at key (seed low, seed high) and counter
// words (counter low, counter high, subsequence low, subsequence high), so the
// first curand4 returns the Philox4x32-10 block of that counter.
#include <curand_kernel.h>

#include <cstdio>
#include <vector>

__global__ void philox_blocks(const unsigned long long *in, uint4 *out, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    curandStatePhilox4_32_10_t st;
    curand_init(in[3 * i], in[3 * i + 1], 4ull * in[3 * i + 2], &st);
    out[i] = curand4(&st);
}

int main()
{
    std::vector<unsigned long long> h;
    unsigned long long a, b, c;
    while (std::scanf("%llu %llu %llu", &a, &b, &c) == 3) {
        h.push_back(a);
        h.push_back(b);
        h.push_back(c);
    }
    const int n = (int)(h.size() / 3);
    if (n == 0)
        return 0;
    unsigned long long *d_in = nullptr;
    uint4 *d_out = nullptr;
    if (cudaMalloc(&d_in, h.size() * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMalloc(&d_out, n * sizeof(uint4)) != cudaSuccess) {
        std::fprintf(stderr, "cudaMalloc failed\n");
        return 1;
    }
    cudaMemcpy(d_in, h.data(), h.size() * sizeof(unsigned long long), cudaMemcpyHostToDevice);
    philox_blocks<<<(n + 127) / 128, 128>>>(d_in, d_out, n);
    std::vector<uint4> r(n);
    if (cudaMemcpy(r.data(), d_out, n * sizeof(uint4), cudaMemcpyDeviceToHost) != cudaSuccess) {
        std::fprintf(stderr, "kernel failed: %s\n", cudaGetErrorString(cudaGetLastError()));
        return 1;
    }
    for (int i = 0; i < n; ++i)
        std::printf("%08x %08x %08x %08x\n", r[i].x, r[i].y, r[i].z, r[i].w);
    cudaFree(d_in);
    cudaFree(d_out);
    return 0;
}
