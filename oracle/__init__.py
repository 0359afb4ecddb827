"""CPU oracle for lattice weight quantization -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 NumPy restatement of what the hot path computes.  Only
the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of the
benchmark may import it; the library under ``lattice_vq_weight_gb300`` never
does, and this package never imports the library.

Parity status of every public function is stated in its docstring; all are
pinned by tests that do not re-derive them (closed forms, textbook constants,
brute force, invariants, hand-worked cases).
"""
from .lattice_oracle import (  # noqa: F401
    LATTICE_DIM,
    LATTICES,
    splitmix64,
    splitmix64_signs,
    hadamard_matrix,
    rht_tiles,
    inverse_rht_tiles,
    round_half_even,
    nearest_z1,
    nearest_dn,
    nearest_e8,
    nearest_a2,
    nearest_point,
    point_to_codes,
    codes_to_point,
    code_membership_ok,
    brute_nearest,
    block_sqdist,
    tile_scales,
    quantize,
    dequantize,
    rht_activations,
    gemv,
    gemm,
    dense_reconstruction_matmul,
    normalized_second_moment,
    covolume,
    compression_ratio,
    pick_tile,
    code_entropy_bits,
    QuantResult,
)
from . import scale_formats  # noqa: F401,E402
