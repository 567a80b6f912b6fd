"""Build libstatekv.so in-tree for sm_103a (GB300) with nvcc.

Usage: python -m kv_cache_compression_frame_gb300.build_lib [--force] [-v]

Each .cu file is compiled to an object in parallel, then linked into one
shared library next to this file.  An object is rebuilt unless the SHA-256
recorded beside it matches its source, every header and the compiler flags;
the library is relinked unless its recorded hash matches its objects'.  A
prebuilt object or library carried in from elsewhere, without the matching
record, is therefore never reused.
"""

from __future__ import annotations

import argparse
import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libstatekv.so")

SOURCES = ["statekv_api.cu", "rope.cu", "attn_tc.cu", "attn_simt.cu", "select.cu",
           "attend_static.cu", "decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                 "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sha(*parts: bytes) -> str:
    h = hashlib.sha256()
    for p in parts:
        h.update(len(p).to_bytes(8, "little"))
        h.update(p)
    return h.hexdigest()


def _read(path: str) -> bytes:
    with open(path, "rb") as f:
        return f.read()


def _headers_digest() -> str:
    hs = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    hs += sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE))
    return _sha(*[os.path.basename(h).encode() + b"\0" + _read(h) for h in hs])


def _stamp_ok(target: str, digest: str) -> bool:
    stamp = target + ".sha"
    return (os.path.exists(target) and os.path.exists(stamp)
            and _read(stamp).decode().strip() == digest)


def _write_stamp(target: str, digest: str) -> None:
    with open(target + ".sha", "w") as f:
        f.write(digest + "\n")


def _compile(nvcc: str, src: str, force: bool, verbose: bool, extra: list[str],
             headers: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    path = os.path.join(CSRC, src)
    cmd = [nvcc, *CFLAGS, *extra, "-c", path, "-o", obj]
    digest = _sha(_read(path), headers.encode(), " ".join([*CFLAGS, *extra]).encode())
    if not force and _stamp_ok(obj, digest):
        return obj, digest
    if verbose:
        print(" ".join(cmd), flush=True)
    if os.path.exists(obj + ".sha"):
        os.remove(obj + ".sha")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    _write_stamp(obj, digest)
    return obj, digest


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    headers = _headers_digest()
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        built = list(ex.map(lambda s: _compile(nvcc, s, force or ptxas_info, verbose, extra,
                                               headers), SOURCES))
    objs = [o for o, _ in built]
    digest = _sha(*[d.encode() for _, d in built], " ".join(ARCH).encode())
    if force or not _stamp_ok(LIB, digest):
        if os.path.exists(LIB + ".sha"):
            os.remove(LIB + ".sha")
        tmp = LIB + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        _write_stamp(LIB, digest)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    a = ap.parse_args()
    print(build(a.force, a.verbose, a.ptxas_info))
    sys.exit(0)
