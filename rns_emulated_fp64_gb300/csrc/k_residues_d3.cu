// Step 2 residue kernels for double entries and N = 17..18 moduli.
#include "k_residues.cuh"

namespace os2dev {

OS2_RESIDUES_PART(residues_d3) {
  switch (N) {
    OS2_RESIDUES_CASE(17, double) OS2_RESIDUES_CASE(18, double)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace os2dev
