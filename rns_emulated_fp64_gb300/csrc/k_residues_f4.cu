// Step 2 residue kernels for float entries and N = 19..20 moduli.
#include "k_residues.cuh"

namespace os2dev {

OS2_RESIDUES_PART(residues_f4) {
  switch (N) {
    OS2_RESIDUES_CASE(19, float) OS2_RESIDUES_CASE(20, float)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace os2dev
