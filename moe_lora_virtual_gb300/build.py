"""Build libmol.so (the MoL LoRA CUDA library) in-tree with nvcc for sm_103a."""

from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG_DIR, "libmol.so")
# The same sources with device-side index checks (MOL_CHECKED): a diagnostic build.
CHECKED_LIB_PATH = os.path.join(PKG_DIR, "libmol_checked.so")

SOURCES = ["mol_abi.cu", "mol_align.cu", "mol_lora.cu", "mol_umma.cu", "mol_stage.cu",
           "mol_expand_tc.cu"]
HEADERS = ["mol_device.cuh", "mol_internal.h", "mol_tc.cuh"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the MoL library needs the CUDA toolkit to build")


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "mol.h"),
                                                                 os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def _command(out: str, checked: bool, verbose: bool) -> list:
    cmd = [nvcc_path(), "-O3", "-std=c++17", *ARCH_FLAGS, "-lineinfo", "-Xcompiler", "-fPIC",
           "-shared", "-I", INCLUDE, "--threads", "4", "-o", out]
    if checked:
        cmd += ["-DMOL_CHECKED"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    return cmd + [os.path.join(CSRC, f) for f in SOURCES]


def build_library(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile the translation units (nvcc --threads 4) into one shared library.

    checked=True builds libmol_checked.so, the same kernels with the device-side
    index checks compiled in."""
    path = CHECKED_LIB_PATH if checked else LIB_PATH
    if not force and not _stale(path):
        return path
    tmp = path + f".tmp{os.getpid()}"
    res = subprocess.run(_command(tmp, checked, verbose), capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, path)
    return path


def build_all(force: bool = False) -> tuple:
    """Build the release and the checked library at the same time (two nvcc processes)."""
    jobs = []
    for checked in (False, True):
        path = CHECKED_LIB_PATH if checked else LIB_PATH
        if force or _stale(path):
            tmp = path + f".tmp{os.getpid()}"
            jobs.append((path, tmp, subprocess.Popen(_command(tmp, checked, False),
                                                     stdout=subprocess.PIPE,
                                                     stderr=subprocess.STDOUT, text=True)))
    errors = []
    for path, tmp, proc in jobs:
        out, _ = proc.communicate()
        if proc.returncode != 0:
            errors.append(f"{os.path.basename(path)}:\n{out}")
        else:
            os.replace(tmp, path)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    return LIB_PATH, CHECKED_LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
