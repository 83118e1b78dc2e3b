"""Build the CUDA library libgbce.so in-tree (cross_entropy_loss_ce_gb300/_lib/).

One translation unit, one -gencode (sm_103a), the CUDA runtime linked
statically; the result exports only the C ABI declared in include/gbce.h.
"""
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "gbce.cu")]


def deps():
    """Every file the library is compiled from: the sources, every header
    under csrc/ and the public headers (a change to any of them rebuilds)."""
    return sorted(set(SOURCES) | set(glob.glob(os.path.join(CSRC, "*.cu")))
                  | set(glob.glob(os.path.join(CSRC, "*.cuh")))
                  | set(glob.glob(os.path.join(ROOT, "include", "*.h"))))


LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libgbce.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "-ftz=true",
    "-Xcompiler", "-fPIC,-fvisibility=hidden", "-shared",
    "-Xptxas", "-v",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libgbce.so unless it is newer than every source; return its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *SOURCES, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(LIB_DIR, "build.log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed (exit {r.returncode}); see {log}")
    if verbose:
        sys.stdout.write(r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


def register_report(log_path: str = None) -> str:
    """Registers, spill stores / loads and static shared memory of every kernel
    instance, one line each, from the -Xptxas -v lines of the last build."""
    import re
    text = open(log_path or os.path.join(LIB_DIR, "build.log")).read()
    rows, cur = [], None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = {"name": m.group(1)}
            rows.append(cur)
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            cur["spill"] = (int(m.group(1)), int(m.group(2)))
        m = re.search(r"Used (\d+) registers.*?(\d+) bytes smem", line)
        if m:
            cur["regs"], cur["smem"] = int(m.group(1)), int(m.group(2))
        elif "Used" in line:
            m = re.search(r"Used (\d+) registers", line)
            if m:
                cur["regs"] = int(m.group(1))
    try:
        names = subprocess.run(["c++filt"], input="\n".join(r["name"] for r in rows),
                               capture_output=True, text=True).stdout.splitlines()
    except OSError:
        names = [r["name"] for r in rows]
    out = [f"{'regs':>4} {'spill st/ld':>11} {'smem':>6}  kernel"]
    for r, name in sorted(zip(rows, names), key=lambda p: p[1]):
        st, ld = r.get("spill", (0, 0))
        out.append(f"{r.get('regs', 0):>4} {f'{st}/{ld}':>11} {r.get('smem', 0):>6}  "
                   + name.replace("gbce::", ""))
    return "\n".join(out)


if __name__ == "__main__":
    if "--registers" in sys.argv:
        print(register_report())
    else:
        print(build(force=True, verbose="-v" in sys.argv))
