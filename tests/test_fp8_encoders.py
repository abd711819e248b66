"""CPU checks of the FP8 GEMM's encoders against the documented bit fields.

The block-scaled FP8 GEMM builds, at compile time, the tcgen05 instruction
descriptor of kind::mxf8f6f4, the shared-memory descriptor of a scale-factor
atom, and the byte position of every UE8M0 scale inside its 512-byte atom. A
host program (tests/host/fp8_encoders.cu, compiled with nvcc, no GPU needed)
prints them; this test rebuilds each value independently:

  * the instruction descriptor field by field from the block-scaled table of
    the PTX ISA (B scale id [4,6), A/B formats [7,10)/[10,13) = E4M3 (0),
    majors [15]/[16], N>>3 in [17,23), UE8M0 scale type bit 23, M>>4 in
    [24,29), A scale id [29,31)); the fields of the bf16 descriptor where the
    two tables agree;
  * the scale-atom descriptor: start>>4 in [0,14), LBO 0, SBO 128>>4 in
    [32,46), version 1 at bit 46, no swizzle;
  * the atom layout through a model of tcgen05.cp .32x128b.warpx4 (line i of
    16 bytes -> lane i, columns 0-3, replicated to lanes 32q+i) and of where
    the block-scaled MMA reads the scale of row r for K block kb (column
    (r % 128) / 32, lane r % 32 of any quarter, byte = scale id = kb % 4):
    every (row, K block) of an atom must come back from its own byte, and no
    two share one.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "routing_dispatch_expert_router_gb300", "csrc")


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


@pytest.fixture(scope="module")
def printed(tmp_path_factory):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("enc") / "fp8_encoders")
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "host", "fp8_encoders.cu"), "-o", exe],
                   check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    rows = {}
    for line in out.splitlines():
        key, *vals = line.split()
        rows.setdefault(key, []).append([int(v) for v in vals])
    return rows


def idesc_model(M, N, a_mn, b_mn, sf_id):
    fields = [  # (value, lsb, width)
        (sf_id, 4, 2),      # scale-factor id of B
        (0, 7, 3),          # A format E4M3
        (0, 10, 3),         # B format E4M3
        (a_mn, 15, 1),
        (b_mn, 16, 1),
        (N >> 3, 17, 6),
        (1, 23, 1),         # scale type UE8M0
        (M >> 4, 24, 5),
        (sf_id, 29, 2),     # scale-factor id of A
    ]
    d = 0
    for v, lsb, w in fields:
        assert 0 <= v < (1 << w)
        d |= v << lsb
    return d


def test_block_scaled_instruction_descriptor(printed):
    for M, N, a_mn, b_mn, sf, got in printed["idesc"]:
        assert got == idesc_model(M, N, a_mn, b_mn, sf), (M, N, a_mn, b_mn, sf)
        # reserved bits 0-1, 3, 6, 31 stay clear; no sparsity, no negation
        assert got & ((1 << 0) | (1 << 1) | (1 << 2) | (1 << 3) | (1 << 6) | (1 << 13) |
                      (1 << 14) | (1 << 31)) == 0


def test_shape_fields_match_the_bf16_descriptor(printed):
    (bf16,), = printed["bf16"]
    mx = [v for *k, v in printed["idesc"] if k == [128, 256, 0, 1, 0]][0]
    for lsb, w in ((15, 1), (16, 1), (17, 6), (24, 5)):
        mask = ((1 << w) - 1) << lsb
        assert bf16 & mask == mx & mask


def test_scale_atom_shared_memory_descriptor(printed):
    for start, d in printed["sfdesc"]:
        assert d & 0x3FFF == (start >> 4) & 0x3FFF
        assert (d >> 16) & 0x3FFF == 0             # LBO: one core matrix along K
        assert (d >> 32) & 0x3FFF == 128 >> 4      # SBO: 8 lines of 16 bytes
        assert (d >> 46) & 0x3 == 1                # descriptor version
        assert (d >> 61) & 0x7 == 0                # no swizzle
        assert d & ~((0x3FFF) | (0x3FFF << 32) | (0x3 << 46)) == 0


def test_scale_atom_layout_through_the_copy_model(printed):
    byte = {(r, kb): b for r, kb, b in printed["atom"]}
    # the copy: atom line i (bytes 16i .. 16i+15) -> lane 32q + i, columns 0..3
    tmem = {}
    for lane in range(128):
        i = lane % 32
        for col in range(4):
            for b in range(4):
                tmem[(lane, col, b)] = 16 * i + 4 * col + b
    seen = set()
    for r in range(128):
        for kb in range(8):
            pos = byte[(r, kb)]
            assert pos == byte[(r, kb % 4)]        # four K blocks per atom, then the next atom
            assert 0 <= pos < 512
            for q in range(4):                     # every lane quarter holds the same bytes
                assert tmem[(32 * q + r % 32, (r % 128) // 32, kb % 4)] == pos
            if kb < 4:
                assert pos not in seen
                seen.add(pos)
    assert len(seen) == 512


def test_atom_counts_and_offsets(printed):
    (a128, a768, a7168), = printed["atoms_k"]
    assert (a128, a768, a7168) == (1, 2, 14)        # ceil(K / 128 / 4)
    (sfb,), = printed["sf_bytes"]
    assert sfb == 163840 // 128 * 14 * 512
    (off,), = printed["atom_offset"]
    assert off == (3 * 14 + 9 // 4) * 512
