// Step 2 residue kernels for float entries and N = 17..18 moduli.
#include "k_residues.cuh"

namespace os2dev {

OS2_RESIDUES_PART(residues_f3) {
  switch (N) {
    OS2_RESIDUES_CASE(17, float) OS2_RESIDUES_CASE(18, float)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace os2dev
