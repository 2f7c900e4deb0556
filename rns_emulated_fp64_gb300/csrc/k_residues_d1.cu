// Step 2 residue kernels for double entries and N = 1..12 moduli.
#include "k_residues.cuh"

namespace os2dev {

OS2_RESIDUES_PART(residues_d1) {
  switch (N) {
    OS2_RESIDUES_CASE(1, double) OS2_RESIDUES_CASE(2, double) OS2_RESIDUES_CASE(3, double) OS2_RESIDUES_CASE(4, double) OS2_RESIDUES_CASE(5, double) OS2_RESIDUES_CASE(6, double) OS2_RESIDUES_CASE(7, double) OS2_RESIDUES_CASE(8, double) OS2_RESIDUES_CASE(9, double) OS2_RESIDUES_CASE(10, double) OS2_RESIDUES_CASE(11, double) OS2_RESIDUES_CASE(12, double)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace os2dev
