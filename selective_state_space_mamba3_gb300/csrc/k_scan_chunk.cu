// Single-pass TF32 instances of the chunked scan (kernel template in
// scan_chunk.cuh) and the host entry points of the chunked path: which shapes
// it takes, and the launch of either flavour.
#include "scan_chunk.cuh"

namespace m3 {

bool chunk_supported(const ScanGeom& g) {
  return (g.R == 1 || g.R == 2 || g.R == 4 || g.R == 8) && g.N <= 128 && g.P <= 128 &&
         g.A <= kAngMax;
}

int chunk_rows_per_token(const ScanGeom& g) { return kRows / g.R; }

// The split flavour doubles every operand tile; it runs where that layout
// fits the device's shared memory per block (227 KB on GB300, also the answer
// without a device). The instance choice mirrors dispatch_chunk.
bool chunk_split_supported(const ScanGeom& g) {
  if (!chunk_supported(g)) return false;
  const bool mimo = g.mimo != 0;
  bool async = false;
  if (!mimo && g.R == 1 && g.P == 64 && g.N == 128 && (g.A == 32 || g.A == 64))
    async = chunk_async(128, g.A);
  else if (mimo && g.R == 4 && g.P == 64 && g.N == 64 && g.A == 32)
    async = chunk_async(64, 32);
  const ChunkLayout lay = chunk_layout(g.N, g.P, g.A, g.R, mimo, async, true);
  int dev = 0, limit = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess ||
      limit <= 0) {
    cudaGetLastError();
    limit = 227 * 1024;
  }
  return chunk_smem_bytes(lay, async, true) <= (size_t)limit;
}

cudaError_t launch_scan_chunk_split(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                                    const ChunkIO& io, bool summary, cudaStream_t s);

cudaError_t launch_scan_chunk(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                              const ChunkIO& io, bool summary, bool split, cudaStream_t s) {
  if (split) return launch_scan_chunk_split(g, a, status, io, summary, s);
  return dispatch_chunk<false>(g, a, status, io, summary, s);
}

}  // namespace m3
