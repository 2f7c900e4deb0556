// Step 2 residue kernels for double entries and N = 13..16 moduli.
#include "k_residues.cuh"

namespace os2dev {

OS2_RESIDUES_PART(residues_d2) {
  switch (N) {
    OS2_RESIDUES_CASE(13, double) OS2_RESIDUES_CASE(14, double) OS2_RESIDUES_CASE(15, double) OS2_RESIDUES_CASE(16, double)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace os2dev
