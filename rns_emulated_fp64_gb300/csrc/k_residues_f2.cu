// Step 2 residue kernels for float entries and N = 13..16 moduli.
#include "k_residues.cuh"

namespace os2dev {

OS2_RESIDUES_PART(residues_f2) {
  switch (N) {
    OS2_RESIDUES_CASE(13, float) OS2_RESIDUES_CASE(14, float) OS2_RESIDUES_CASE(15, float) OS2_RESIDUES_CASE(16, float)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace os2dev
