// Split-operand (3xTF32) instances of the chunked scan: the kernel template of
// scan_chunk.cuh with every operand carried as a high and a low TF32 part and
// three MMAs per product, in a translation unit of its own so that the two
// flavours compile in parallel.
#include "scan_chunk.cuh"

namespace m3 {

cudaError_t launch_scan_chunk_split(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                                    const ChunkIO& io, bool summary, cudaStream_t s) {
  return dispatch_chunk<true>(g, a, status, io, summary, s);
}

}  // namespace m3
