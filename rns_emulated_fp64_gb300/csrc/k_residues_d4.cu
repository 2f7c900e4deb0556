// Step 2 residue kernels for double entries and N = 19..20 moduli.
#include "k_residues.cuh"

namespace os2dev {

OS2_RESIDUES_PART(residues_d4) {
  switch (N) {
    OS2_RESIDUES_CASE(19, double) OS2_RESIDUES_CASE(20, double)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace os2dev
