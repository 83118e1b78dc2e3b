"""The in-tree build notices a change to any file the library is compiled
from (CPU only: nvcc cross-compiles sm_103a without a GPU)."""
import os

from cross_entropy_loss_ce_gb300 import build as gbuild


def test_every_kernel_header_is_a_dependency():
    names = {os.path.basename(p) for p in gbuild.deps()}
    on_disk = {f for f in os.listdir(gbuild.CSRC) if f.endswith((".cu", ".cuh"))}
    assert on_disk <= names
    assert "gbce.h" in names


def test_touching_a_kernel_header_makes_the_library_stale():
    lib = gbuild.build()
    assert gbuild.up_to_date()
    t_lib = os.path.getmtime(lib)
    for name in ("bsr_kernels.cuh", "row_kernels.cuh", "device.cuh"):
        path = os.path.join(gbuild.CSRC, name)
        st = os.stat(path)
        try:
            os.utime(path, (st.st_atime, t_lib + 10))
            assert not gbuild.up_to_date(), f"an edit to {name} would not rebuild the library"
        finally:
            os.utime(path, (st.st_atime, st.st_mtime))
    assert gbuild.up_to_date()
