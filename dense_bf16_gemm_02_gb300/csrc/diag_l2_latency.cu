// Diagnostic program (not part of the library): L2-hit latency by SM and by
// address region, the evidence behind the grid schedule's die question. Each
// CTA (one per SM) walks a pointer chain of distinct 128-byte lines inside each
// of R regions of an L2-resident buffer and records the average cycles per
// load, with its %smid; a near/far split between the two dies' L2 halves would
// show as SMs whose latencies differ by region. Read-only after set-up; every
// index stays inside its region. Prints one line per CTA: smid and R latencies.
#include <cstdio>
#include <cstdint>
#include <vector>
#include <algorithm>
#include <cuda_runtime.h>
#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("%s: %s\n", #x, cudaGetErrorString(e)); return 1; } } while (0)
constexpr int R = 32;              // regions
constexpr int kRegionWords = 1 << 18;   // 1 MiB of uint32 per region
constexpr int kHops = 128;
__global__ void probe(const uint32_t* __restrict__ buf, uint32_t* smid_out, float* lat_out) {
    if (threadIdx.x != 0) return;
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    smid_out[blockIdx.x] = smid;
    for (int r = 0; r < R; ++r) {
        const uint32_t* reg = buf + (size_t)r * kRegionWords;
        uint32_t idx = 0;
        for (int h = 0; h < kHops; ++h) idx = __ldcg(reg + idx);            // warm (L2)
        long long t0 = clock64();
        for (int h = 0; h < kHops; ++h) idx = __ldcg(reg + idx);
        long long t1 = clock64();
        lat_out[blockIdx.x * R + r] = float(t1 - t0) / kHops + (idx == 0xFFFFFFFFu ? 1.0f : 0.0f);
    }
}
int main() {
    int sms = 0; CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
    std::vector<uint32_t> h((size_t)R * kRegionWords);
    // a chain of kHops + 1 distinct 128-byte lines per region (indices stay in the region)
    uint64_t x = 88172645463325252ull;
    for (int r = 0; r < R; ++r) {
        std::vector<uint32_t> lines;
        for (int i = 0; i < kHops + 1; ++i) { x ^= x << 13; x ^= x >> 7; x ^= x << 17; lines.push_back((uint32_t)((x % (kRegionWords / 32)) * 32)); }
        std::sort(lines.begin(), lines.end()); lines.erase(std::unique(lines.begin(), lines.end()), lines.end());
        uint32_t* reg = h.data() + (size_t)r * kRegionWords;
        reg[0] = lines[0];
        for (size_t i = 0; i + 1 < lines.size(); ++i) reg[lines[i]] = lines[i + 1];
        reg[lines.back()] = lines[0];
    }
    uint32_t* d = nullptr; uint32_t* smid = nullptr; float* lat = nullptr;
    CK(cudaMalloc(&d, h.size() * 4)); CK(cudaMalloc(&smid, sms * 4)); CK(cudaMalloc(&lat, sms * R * 4));
    CK(cudaMemcpy(d, h.data(), h.size() * 4, cudaMemcpyHostToDevice));
    for (int rep = 0; rep < 2; ++rep) probe<<<sms, 32>>>(d, smid, lat);
    CK(cudaGetLastError()); CK(cudaDeviceSynchronize());
    std::vector<uint32_t> hs(sms); std::vector<float> hl(sms * R);
    CK(cudaMemcpy(hs.data(), smid, sms * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(hl.data(), lat, sms * R * 4, cudaMemcpyDeviceToHost));
    for (int b = 0; b < sms; ++b) {
        printf("smid %3u:", hs[b]);
        for (int r = 0; r < R; ++r) printf(" %5.0f", hl[b * R + r]);
        printf("\n");
    }
    return 0;
}
