// Step 2 residue kernels for float entries and N = 1..12 moduli.
#include "k_residues.cuh"

namespace os2dev {

OS2_RESIDUES_PART(residues_f1) {
  switch (N) {
    OS2_RESIDUES_CASE(1, float) OS2_RESIDUES_CASE(2, float) OS2_RESIDUES_CASE(3, float) OS2_RESIDUES_CASE(4, float) OS2_RESIDUES_CASE(5, float) OS2_RESIDUES_CASE(6, float) OS2_RESIDUES_CASE(7, float) OS2_RESIDUES_CASE(8, float) OS2_RESIDUES_CASE(9, float) OS2_RESIDUES_CASE(10, float) OS2_RESIDUES_CASE(11, float) OS2_RESIDUES_CASE(12, float)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace os2dev
