"""Build libsinkattn.so (the CUDA kernels plus the C ABI) for sm_103a with nvcc.

Translation units are compiled in parallel into _build/, then linked into
paged_gqa_attention_head_gb300/libsinkattn.so.  `python -m
paged_gqa_attention_head_gb300.build` runs it; __graft_entry__.build() calls it.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsinkattn.so")
SOURCES = ["api.cpp", "decode.cu", "decode_fp8.cu", "append.cu", "prefill.cu", "decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")


# The prefill kernel re-balances registers between warpgroups with setmaxnreg; the
# split adds up to exactly the registers it is launched with (512 threads x 128), so
# the build refuses any other register count (a larger split than the launch
# budget would make setmaxnreg wait forever).
PREFILL_LAUNCH_REGS = 128


def _check_prefill_regs(ptxas_log: str) -> None:
    fn = None
    found = 0
    for line in ptxas_log.splitlines():
        if "Compiling entry function" in line:
            fn = line
        elif "Used" in line and "registers" in line and fn and "prefill_kernel" in fn:
            regs = int(line.split("Used")[1].split("registers")[0])
            found += 1
            if regs != PREFILL_LAUNCH_REGS:
                raise RuntimeError(f"prefill_kernel uses {regs} registers, expected "
                                   f"{PREFILL_LAUNCH_REGS} (its setmaxnreg split depends on it)")
            fn = None
    if found == 0:
        raise RuntimeError("ptxas did not report the prefill kernel's registers")


def _flags(extra_ptxas_verbose: bool) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "--expt-relaxed-constexpr", "-I", os.path.join(HERE, "..", "include")]
    if extra_ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(HERE, "..", "include", "sinkattn.h"))
    newest = max(os.path.getmtime(p) for p in deps)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        is_prefill = os.path.basename(src) == "prefill.cu"
        cmd = [NVCC, "-c", src, "-o", obj] + _flags(verbose or is_prefill)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if is_prefill:
            _check_prefill_regs(r.stderr)
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
