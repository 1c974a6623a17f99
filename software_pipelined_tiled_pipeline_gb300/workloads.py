"""The synthetic GEMM workloads the library is measured and checked on.

Shapes, layouts, element types and value distributions follow the square
synthetic GEMMs in "CUDA Kernel Study: Pipelining" (Kernel Parameters),
"pipeline-gpu-kernel" (Step 2, the 4096^3 IGEMM) and "Part 4 -- Pipelining and
Occupancy" (section 4.3, the 4096^3 FP32 sweep), widened to the stage/ratio
sweep.  Operands come from ``synth`` with the base seed below.
"""
from dataclasses import dataclass, field
from typing import Tuple

BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "i8" | "f16" | "bf16" | "f32"
    layout: str           # "row_col" | "row_row"
    M: int
    N: int
    K: int
    stages: Tuple[int, ...] = field(default=(2,))
    variants: Tuple[str, ...] = field(default=("pipelined", "pingpong"))
    description: str = ""

    @property
    def ops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def read_bytes(self) -> int:
        """A and B, read once."""
        return (self.M + self.N) * self.K * {"i8": 1, "f16": 2, "bf16": 2, "f32": 4}[self.dtype]

    @property
    def write_bytes(self) -> int:
        """C, written once."""
        return self.M * self.N * {"i8": 4, "f16": 2, "bf16": 2, "f32": 4}[self.dtype]

    @property
    def algorithmic_bytes(self) -> int:
        """A and B read once, C written once: the least DRAM traffic of one GEMM."""
        size_in = {"i8": 1, "f16": 2, "bf16": 2, "f32": 4}[self.dtype]
        size_out = {"i8": 4, "f16": 2, "bf16": 2, "f32": 4}[self.dtype]
        return (self.M + self.N) * self.K * size_in + self.M * self.N * size_out


WORKLOADS = {
    w.name: w for w in [
        Workload("i8_256", "i8", "row_col", 256, 256, 256, (2, 3, 4), ("pipelined", "pingpong", "nopipe"),
                 "INT8 GEMM M=N=K=256, A row-major, B column-major, uniform int8, INT32 out"),
        Workload("f32_1024", "f32", "row_row", 1024, 1024, 1024, (2, 3, 4), ("pipelined", "pingpong", "nopipe"),
                 "FP32 SGEMM M=N=K=1024 on the FFMA path, row-major, U[-1,1]"),
        Workload("i8_4096", "i8", "row_col", 4096, 4096, 4096, (2, 3, 4, 6), ("pipelined", "pingpong", "nopipe"),
                 "INT8 IGEMM M=N=K=4096, A row-major, B column-major, uniform int8, INT32 out"),
        Workload("f16_4096", "f16", "row_col", 4096, 4096, 4096, (2, 3, 4, 5, 6), ("pipelined", "pingpong", "nopipe"),
                 "FP16 GEMM M=N=K=4096, A row-major, B column-major, U[-1,1], FP32 accumulate, FP16 out"),
        Workload("bf16_8192_k256", "bf16", "row_col", 8192, 8192, 256, tuple(range(2, 9))),
        Workload("bf16_8192_k1024", "bf16", "row_col", 8192, 8192, 1024, tuple(range(2, 9))),
        Workload("bf16_8192_k4096", "bf16", "row_col", 8192, 8192, 4096, tuple(range(2, 9))),
        Workload("bf16_8192_k16384", "bf16", "row_col", 8192, 8192, 16384, tuple(range(2, 9))),
        Workload("f32_4096", "f32", "row_row", 4096, 4096, 4096, (3,), ("pipelined",),
                 "FP32 SGEMM M=N=K=4096 on the FFMA path (the register-tile sweep's size)"),
        Workload("bf16_skinny", "bf16", "row_col", 8192, 128, 8192, tuple(range(2, 9)),
                 description="BF16 low compute/load ratio case M=8192, N=128, K=8192"),
    ]
}
