"""Builds the sm_103a shared libraries in-tree with nvcc.

  libmoe_b300.so    the MoE layer (routed_expert_ffn_bucketing_b300/csrc) behind include/moe.h
  libsynth_b300.so  the device half of the seeded input generator (synth/csrc)

Objects go to _build/ at the repository root, and a source is rebuilt when it or any header
next to it is newer than its object. Run as `python -m routed_expert_ffn_bucketing_b300.build`.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]

LIBS = {
    "moe": dict(src_dir=os.path.join(PKG, "csrc"), out=os.path.join(PKG, "libmoe_b300.so"),
                inc=[os.path.join(ROOT, "include")]),
    "synth": dict(src_dir=os.path.join(ROOT, "synth", "csrc"), out=os.path.join(ROOT, "synth", "libsynth_b300.so"),
                  inc=[]),
}


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _newest(paths):
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def _compile(src: str, obj: str, inc: list[str], deps: list[str], verbose: bool) -> str:
    if os.path.exists(obj) and os.path.getmtime(obj) >= _newest([src] + deps):
        return obj
    cmd = [nvcc()] + NVCC_FLAGS + [f"-I{d}" for d in inc] + ["-c", src, "-o", obj]
    if src.endswith(".cpp"):
        cmd = [nvcc()] + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O3,-fopenmp"] + [f"-I{d}" for d in inc] + \
            ["-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build_lib(name: str, verbose: bool = False) -> str:
    cfg = LIBS[name]
    src_dir = cfg["src_dir"]
    srcs = sorted(os.path.join(src_dir, f) for f in os.listdir(src_dir) if f.endswith((".cu", ".cpp")))
    hdrs = [os.path.join(src_dir, f) for f in os.listdir(src_dir) if f.endswith((".h", ".cuh"))]
    for d in cfg["inc"]:
        hdrs += [os.path.join(d, f) for f in os.listdir(d) if f.endswith(".h")]
    odir = os.path.join(BUILD, name)
    os.makedirs(odir, exist_ok=True)
    objs = [os.path.join(odir, os.path.basename(s) + ".o") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        list(ex.map(lambda so: _compile(so[0], so[1], cfg["inc"], hdrs, verbose), zip(srcs, objs)))
    out = cfg["out"]
    if not (os.path.exists(out) and os.path.getmtime(out) >= _newest(objs)):
        cmd = [nvcc()] + ARCH + ["-shared", "-o", out] + objs + ["-lcudart_static", "-lrt", "-ldl", "-lpthread", "-lgomp"]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {out} failed:\n{r.stdout}\n{r.stderr}")
    return out


def build_all(verbose: bool = False) -> list[str]:
    return [build_lib(n, verbose) for n in LIBS]


if __name__ == "__main__":
    for p in build_all(verbose="-v" in sys.argv):
        print(p)
