// Checks the reporting path of the bounds-checked build (MOEFFN_BOUNDS_CHECK):
// in_bounds accepts indices in [0, n), and for one outside it sets the
// DEV_ERR_BOUNDS bit and records the first site and index only.  No access
// is made with any index here.  Prints "code <c> where <w> index <i> ok <n>".
#include "common.cuh"

#include <cstdio>

using moeffn::DevStatus;
using moeffn::in_bounds;

__global__ void probe(DevStatus* st, int* ok) {
    int n = 0;
    n += in_bounds(st, 0, 3, 11);
    n += in_bounds(st, 2, 3, 12);
    n += !in_bounds(st, 5, 3, 42);        // first failure: recorded
    n += !in_bounds(st, -1, 3, 43);       // later failures leave the record as it is
    n += in_bounds(st, 7, 8, 44);
    *ok = n;
}

int main() {
    DevStatus* st;
    int* ok;
    if (cudaMalloc(&st, sizeof(DevStatus)) != cudaSuccess || cudaMalloc(&ok, sizeof(int)) != cudaSuccess) return 2;
    cudaMemset(st, 0, sizeof(DevStatus));
    probe<<<1, 1>>>(st, ok);
    if (cudaDeviceSynchronize() != cudaSuccess) return 3;
    DevStatus h;
    int hok = 0;
    cudaMemcpy(&h, st, sizeof(h), cudaMemcpyDeviceToHost);
    cudaMemcpy(&hok, ok, sizeof(int), cudaMemcpyDeviceToHost);
    std::printf("code %u where %u index %u ok %d\n", h.code, h.bounds_where, h.bounds_index, hok);
    return 0;
}
