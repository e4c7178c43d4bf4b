"""The C-ABI library without a GPU: it builds, loads, exports exactly what the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from sparse_attention_key_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lightning_indexer.h")


@pytest.fixture(scope="module")
def L():
    path = lib_build.build()
    from sparse_attention_key_gb300 import binding
    return binding.lib() if binding.library_path() == path else ctypes.CDLL(path)


def declared_functions():
    src = open(HEADER).read()
    return re.findall(r"IDX_API\s+[\w\s\*]+?\b(idx_\w+)\s*\(", src)


def test_header_declares_the_api():
    names = declared_functions()
    assert {"idx_key_layernorm", "idx_score", "idx_topk", "idx_score_topk"} <= set(names)
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_library_exports_nothing_else():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib_build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.split()[1] in ("T", "t")}
    assert exported == set(declared_functions())


def test_binding_export_list_matches_header():
    from sparse_attention_key_gb300 import binding
    assert set(binding.EXPORTS) == set(declared_functions())


def test_version(L):
    from sparse_attention_key_gb300 import binding
    assert binding.version() >= 100


def test_workspace_sizes_are_host_only(L):
    from sparse_attention_key_gb300 import binding
    assert binding.topk_workspace_size(10, 5000, 2048) >= 256
    s = binding.score_topk_workspace_size(4, 3200, 50800, 2048)
    assert s >= 3200 * 50800 * 4
    assert s % 256 == 0
    # arguments the calls reject: the header size, not a wrapped-around count
    assert binding.score_topk_workspace_size(0, 3200, 50800, 2048) == 256
    assert binding.score_topk_workspace_size(4, -1, 50800, 2048) == 256
    assert binding.score_topk_workspace_size(4, 3200, 0, 2048) == 256
    assert binding.topk_workspace_size(-1, 50800, 2048) == 256
    L.idx_score_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64]
    L.idx_score_workspace_size.restype = ctypes.c_size_t
    assert L.idx_score_workspace_size(0, 10, 100) == 256
    assert L.idx_score_workspace_size(2, -3, 100) == 256
    assert L.idx_score_workspace_size(2, 10, 100) > 256


# Host argument errors: each returns its code with no CUDA call (no GPU here).
FAKE = ctypes.c_void_p(4096)      # a non-null, aligned, never dereferenced address
NULL = None


def _score_topk(L, **kw):
    a = dict(q=FAKE, k=FAKE, w=FAKE, q_pos=FAKE, cu_q=FAKE, cu_k=FAKE, B=1, T=4, n_keys=100,
             max_len=100, topk=2048, idx=FAKE, cnt=NULL, ws=FAKE, ws_bytes=1 << 30, stream=NULL)
    a.update(kw)
    return L.idx_score_topk(a["q"], a["k"], a["w"], a["q_pos"], a["cu_q"], a["cu_k"], a["B"],
                            a["T"], a["n_keys"], a["max_len"], a["topk"], a["idx"], a["cnt"],
                            a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=NULL), 1), (dict(k=NULL), 1), (dict(w=NULL), 1), (dict(q_pos=NULL), 1),
    (dict(cu_q=NULL), 1), (dict(cu_k=NULL), 1), (dict(idx=NULL), 1),
    (dict(B=0), 1), (dict(T=-1), 1), (dict(max_len=0), 1), (dict(topk=0), 1), (dict(n_keys=-1), 1),
    (dict(topk=2049), 1), (dict(q=ctypes.c_void_p(4098)), 1),
    (dict(ws=NULL), 3), (dict(ws_bytes=16), 3), (dict(ws=ctypes.c_void_p(4096 + 16)), 3),
])
def test_score_topk_host_errors(L, kw, code):
    assert _score_topk(L, **kw) == code
    assert L.idx_last_error()  # a message is set


def test_topk_host_errors(L):
    ok = dict(scores=FAKE, ld=4096, n_valid=FAKE, T=3, max_len=4000, topk=16, idx=FAKE,
              cnt=NULL, ws=FAKE, ws_bytes=1 << 20, stream=NULL)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return L.idx_topk(a["scores"], a["ld"], a["n_valid"], a["T"], a["max_len"], a["topk"],
                          a["idx"], a["cnt"], a["ws"], a["ws_bytes"], a["stream"])
    assert call(ld=4098) == 1          # not a multiple of 4
    assert call(topk=0) == 1
    assert call(topk=4096) == 1
    assert call(scores=NULL) == 1
    assert call(n_valid=NULL) == 1
    assert call(ws_bytes=8) == 3
    assert call(T=-2) == 1


def test_score_host_errors(L):
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, w=FAKE, q_pos=FAKE, cu_q=FAKE, cu_k=FAKE, B=1, T=2, n_keys=64,
                 max_len=64, scores=FAKE, ld=64, ws=FAKE, ws_bytes=1 << 20, stream=NULL)
        a.update(kw)
        return L.idx_score(a["q"], a["k"], a["w"], a["q_pos"], a["cu_q"], a["cu_k"], a["B"],
                           a["T"], a["n_keys"], a["max_len"], a["scores"], a["ld"], a["ws"],
                           a["ws_bytes"], a["stream"])
    assert call(ld=60) == 1            # ld < max_len
    assert call(ld=66) == 1            # not a multiple of 4
    assert call(scores=NULL) == 1
    assert call(ws=NULL) == 3


def test_layernorm_host_errors(L):
    def call(**kw):
        a = dict(k_raw=FAKE, w=FAKE, b=FAKE, dt=0, eps=1e-6, out=FAKE, n=10, stream=NULL)
        a.update(kw)
        return L.idx_key_layernorm(a["k_raw"], a["w"], a["b"], a["dt"], ctypes.c_float(a["eps"]),
                                   a["out"], a["n"], a["stream"])
    assert call(n=-1) == 1
    assert call(dt=7) == 1
    assert call(eps=float("nan")) == 1
    assert call(k_raw=NULL) == 1
    assert call(n=0) == 0             # nothing to do: no device needed


def test_layernorm_append_host_errors(L):
    fn = L.idx_key_layernorm_append
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_float, ctypes.c_void_p,
                                           ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                           ctypes.c_void_p]

    def call(**kw):
        a = dict(k_raw=FAKE, w=FAKE, b=FAKE, dt=0, eps=1e-6, cache=FAKE, rows=100, slot=FAKE, n=10)
        a.update(kw)
        return fn(a["k_raw"], a["w"], a["b"], a["dt"], a["eps"], a["cache"], a["rows"], a["slot"],
                  a["n"], NULL)
    assert call(n=-1) == 1
    assert call(rows=-1) == 1
    assert call(dt=3) == 1
    assert call(slot=NULL) == 1
    assert call(cache=NULL) == 1
    assert call(slot=ctypes.c_void_p(4096 + 4)) == 1   # int64 slots: 8-byte aligned
    assert call(n=0) == 0                               # nothing to do: no device needed


def test_indexer_project_host_errors(L):
    fn = L.idx_indexer_project
    P = ctypes.c_void_p
    fn.argtypes = [P] * 7 + [ctypes.c_int, ctypes.c_float, ctypes.c_int32, ctypes.c_int32,
                             ctypes.c_int32, P, P, ctypes.c_int64, P, P, P, ctypes.c_size_t, P]
    L.idx_indexer_project_workspace_size.argtypes = [ctypes.c_int32]
    L.idx_indexer_project_workspace_size.restype = ctypes.c_size_t
    need = L.idx_indexer_project_workspace_size(4)
    assert need >= 4 * 256

    def call(**kw):
        a = dict(T=4, hidden=7168, rank=1536, dt=0, ws_bytes=need, ws=FAKE, x=FAKE)
        a.update(kw)
        return fn(a["x"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["dt"], 1e-6, a["T"], a["hidden"],
                  a["rank"], FAKE, FAKE, 100, FAKE, FAKE, a["ws"], a["ws_bytes"], NULL)
    assert call(hidden=7170) == 1       # not a multiple of 8
    assert call(rank=0) == 1
    assert call(T=-1) == 1
    assert call(dt=5) == 1
    assert call(x=NULL) == 1
    assert call(ws_bytes=need - 1) == 3
    assert call(ws=ctypes.c_void_p(4096 + 16)) == 3
    assert call(T=0) == 0


def test_sparse_mla_host_errors(L):
    fn = L.idx_sparse_mla
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [P, P, ctypes.c_int64, P, P, P, P, i32, i32, i32, i32, ctypes.c_float, P, P, P,
                   ctypes.c_size_t, P]
    L.idx_sparse_mla_workspace_size.argtypes = [i32, i32, i32]
    L.idx_sparse_mla_workspace_size.restype = ctypes.c_size_t
    need = L.idx_sparse_mla_workspace_size(8, 96, 2048)
    assert need >= 256 and need % 256 == 0
    assert L.idx_sparse_mla_workspace_size(8, 48, 2048) == 256   # unsupported heads: header only

    def call(**kw):
        a = dict(q=FAKE, cache=FAKE, rows=1000, idx=FAKE, cnt=FAKE, cu_q=FAKE, cu_k=FAKE, B=1, T=8,
                 H=96, topk=2048, scale=0.07, out=FAKE, lse=FAKE, ws=FAKE, ws_bytes=need)
        a.update(kw)
        return fn(a["q"], a["cache"], a["rows"], a["idx"], a["cnt"], a["cu_q"], a["cu_k"], a["B"],
                  a["T"], a["H"], a["topk"], a["scale"], a["out"], a["lse"], a["ws"], a["ws_bytes"],
                  NULL)
    assert call(H=48) == 1
    assert call(H=128) == 1
    assert call(topk=0) == 1
    assert call(topk=2049) == 1
    assert call(scale=0.0) == 1
    assert call(scale=float("inf")) == 1
    assert call(B=0) == 1
    assert call(T=-1) == 1
    assert call(rows=-5) == 1
    assert call(q=NULL) == 1
    assert call(idx=NULL) == 1
    assert call(cu_k=NULL) == 1
    assert call(out=ctypes.c_void_p(4096 + 4)) == 1   # out must be 16-byte aligned
    assert call(ws=NULL) == 3
    assert call(ws=ctypes.c_void_p(4096 + 16)) == 3
    assert L.idx_last_error()


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from sparse_attention_key_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "lightning_indexer.h"

/* host buffers with the alignment the API asks of device pointers; the calls
   below are rejected before anything is read from them */
#define ALIGNED __attribute__((aligned(256)))
static uint16_t qbuf[256] ALIGNED, kbuf[256] ALIGNED;
static float wbuf[128] ALIGNED;
static int32_t q_pos[1], cu[2] = {0, 1}, idx[IDX_TOPK_MAX];

int main(void) {
    size_t ws = idx_score_topk_workspace_size(1, 1, 1, IDX_TOPK_MAX);
    idx_status s;
    if (idx_version() < 100 || ws < 256 || ws % 256 != 0) return 1;
    /* a misaligned query array: an argument error */
    s = idx_score_topk(qbuf + 1, kbuf, wbuf, q_pos, cu, cu, 1, 1, 1, 1, IDX_TOPK_MAX, idx, NULL,
                       NULL, ws, NULL);
    if (s != IDX_ERR_INVALID_ARG || idx_last_error() == NULL || strlen(idx_last_error()) == 0) return 2;
    /* a null workspace: a workspace error */
    s = idx_score_topk(qbuf, kbuf, wbuf, q_pos, cu, cu, 1, 1, 1, 1, IDX_TOPK_MAX, idx, NULL,
                       NULL, ws, NULL);
    if (s != IDX_ERR_WORKSPACE || strlen(idx_last_error()) == 0) return 3;
    printf("ok %d %zu\n", (int)idx_version(), ws);
    return 0;
}
"""


@pytest.mark.parametrize("lang", ["c99", "c++17"])
def test_plain_c_client_compiles_links_and_runs(tmp_path, lang):
    """The header is valid C and C++ on its own, and a program built with the
    host compiler (no CUDA headers, no torch) links the library and calls it."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c99" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    path = lib_build.build()
    src = tmp_path / ("client.c" if lang == "c99" else "client.cpp")
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    flags = ["-std=" + lang, "-Wall", "-Wextra", "-pedantic", "-Werror"]
    subprocess.run([cc, *flags, "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                    path, "-Wl,-rpath," + os.path.dirname(path)], check=True, capture_output=True,
                   text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")
