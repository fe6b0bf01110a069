// The chunked SISO scan reading the packed input projection directly (the
// preprocess fused into the scan's staging), both flavours: the B / C rows
// arrive by TMA from their columns of the packed rows and are RMS-normalised in
// shared memory, dt and adt are formed from dt_raw / a_raw as the preprocess
// forms them, and x / z are read from their column slices; the outputs have
// the bits of m3_preprocess followed by the scan.
#include "scan_chunk.cuh"

namespace m3 {

bool chunk_packed_supported(const ScanGeom& g) { return packed_instance(g); }

cudaError_t launch_scan_chunk_packed(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                                     const ChunkIO& io, bool summary, bool split,
                                     cudaStream_t s) {
  return split ? dispatch_chunk_packed<true>(g, a, status, io, summary, s)
               : dispatch_chunk_packed<false>(g, a, status, io, summary, s);
}

}  // namespace m3
