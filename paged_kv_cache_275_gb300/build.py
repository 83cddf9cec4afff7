"""Build libpagedkv.so in-tree with nvcc for sm_103a (GB300).

    python -m paged_kv_cache_275_gb300.build [--force] [--ptxas-verbose]

Each CUDA translation unit is compiled in parallel to ``_build/*.o`` and the
objects are linked into ``paged_kv_cache_275_gb300/libpagedkv.so`` against the
shared CUDA runtime.  Rebuilds only when a source or header is newer than the
library.  No cmake, no torch extension machinery.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = PKG / "libpagedkv.so"
SOURCES = ["capi.cu", "kv_append.cu", "paged_decode.cu", "static_workspace.cu", "copy_blocks.cu",
           "block_manager.cpp", "paged_prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> Path:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env:
        return Path(env)
    nvcc = shutil.which("nvcc")
    if nvcc:
        return Path(nvcc).resolve().parent.parent
    return Path("/usr/local/cuda")


def _nvcc() -> str:
    exe = cuda_home() / "bin" / "nvcc"
    return str(exe) if exe.exists() else "nvcc"


def _inputs() -> list[Path]:
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h")) + [Path(__file__)]


STAMP = BUILD / "flags.txt"


def extra_flags() -> list[str]:
    """Extra nvcc flags from PKV_NVCC_FLAGS (launch-shape tuning, e.g. -DPKV_D128_WARPS=6)."""
    return os.environ.get("PKV_NVCC_FLAGS", "").split()


def needs_build() -> bool:
    if not LIB.exists():
        return True
    if (STAMP.read_text() if STAMP.exists() else "") != " ".join(extra_flags()):
        return True
    t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > t for p in _inputs())


def compile_flags(ptxas_verbose: bool = False) -> list[str]:
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", str(INCLUDE), "-I", str(CSRC),
                    "--expt-relaxed-constexpr"] + extra_flags()
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    return flags


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = False) -> Path:
    if not force and not ptxas_verbose and not needs_build():
        return LIB
    BUILD.mkdir(exist_ok=True)
    nvcc = _nvcc()
    flags = compile_flags(ptxas_verbose)

    def one(src: str):
        obj = BUILD / (Path(src).stem + ".o")
        cmd = [nvcc, *flags, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(one, SOURCES))
    for src, _, r in results:
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"nvcc failed on {src}")
        if (ptxas_verbose or r.stderr.strip()) and not quiet:
            sys.stderr.write(r.stderr)
    tmp = LIB.with_name(f"libpagedkv.so.tmp{os.getpid()}")
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", str(tmp), *[str(o) for _, o, _ in results],
            "-Xlinker", f"-rpath,{cuda_home() / 'lib64'}"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, LIB)
    STAMP.write_text(" ".join(extra_flags()))
    return LIB


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true", help="print registers / spills / shared memory")
    args = ap.parse_args(argv)
    print(build(force=args.force, ptxas_verbose=args.ptxas_verbose))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
