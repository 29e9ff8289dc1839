"""Build libtreeverify.so in-tree with nvcc for sm_103a (no GPU needed), and
its bounds-checked twin libtreeverify_checked.so (the same sources compiled
with -DTV_CHECKED: every computed index is checked before the access it
guards, and a failed check is recorded instead of made)."""
from __future__ import annotations

import os
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libtreeverify.so")
CHECKED_LIB_PATH = os.path.join(PKG, "libtreeverify_checked.so")

SOURCES = ["tv_api.cu", "tv_tree.cu", "tv_greedy.cu", "tv_sample.cu", "tv_expand.cu",
           "tv_attn.cu", "tv_commit.cu", "tv_expected.cu", "tv_topn.cu", "tv_spine.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE,
              "-I" + CSRC, "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "treeverify.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _variants(force: bool):
    """(output library, object folder, extra flags) of each build to make."""
    out = []
    for lib, sub, extra in ((LIB_PATH, "", []),
                            (CHECKED_LIB_PATH, "checked", ["-DTV_CHECKED"])):
        if force or not up_to_date(lib):
            out.append((lib, os.path.join(BUILD_DIR, sub) if sub else BUILD_DIR, extra))
    return out


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every source of both builds in parallel, then link each library."""
    todo = _variants(force)
    if not todo:
        return LIB_PATH
    nvcc = _nvcc()
    procs = []
    links = []
    for lib, obj_dir, extra in todo:
        os.makedirs(obj_dir, exist_ok=True)
        objs = []
        for src in SOURCES:
            obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
            objs.append(obj)
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
        links.append((lib, objs))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            print(out)
        if p.returncode != 0:
            errors.append(f"--- {src} ---\n{out}")
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    for lib, objs in links:
        fd, tmp = tempfile.mkstemp(suffix=".so", dir=PKG)
        os.close(fd)
        link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            os.unlink(tmp)
            raise RuntimeError("link failed:\n" + r.stdout)
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
