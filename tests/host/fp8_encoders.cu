// Host program for tests/test_fp8_encoders.py: prints the values of the FP8
// GEMM's compile-time encoders (instruction descriptors, the scale-factor
// shared-memory descriptor and the scale-atom byte layout) so that the test can
// compare them with the documented bit fields and a model of the copy into
// tensor memory. Runs on the CPU only; no kernel is launched.
#include <stdio.h>

#include "fp8_layout.cuh"
#include "ptx.cuh"

int main() {
  using namespace moe;
  const int shapes[][4] = {{128, 256, 0, 0}, {128, 256, 0, 1}, {128, 128, 0, 0}, {64, 64, 1, 1}};
  for (const auto& s : shapes)
    for (unsigned id = 0; id < 4; ++id)
      printf("idesc %d %d %d %d %u %u\n", s[0], s[1], s[2], s[3], id,
             ptx::idesc_with_sf_id(ptx::idesc_mxf8_e4m3(s[0], s[1], s[2], s[3]), id));
  printf("bf16 %u\n", ptx::idesc_bf16(128, 256, 0, 1));
  const unsigned starts[] = {0u, 512u, 1536u, 200704u};
  for (unsigned a : starts)
    printf("sfdesc %u %llu\n", a, (unsigned long long)ptx::smem_desc_sf(a));
  for (int r = 0; r < 128; ++r)
    for (int kb = 0; kb < 8; ++kb) printf("atom %d %d %d\n", r, kb, f8::atom_byte(r, kb));
  printf("atoms_k %lld %lld %lld\n", (long long)f8::atoms_k(128), (long long)f8::atoms_k(768),
         (long long)f8::atoms_k(7168));
  printf("sf_bytes %lld\n", (long long)f8::sf_bytes(163840, 7168));
  printf("atom_offset %lld\n", (long long)f8::atom_offset(3, 9, 14));
  return 0;
}
