"""CPU checks of the C-ABI boundary: the library builds and loads, exports every
function include/m3s.h declares, and rejects bad arguments on the host before
any launch (these calls never reach the GPU)."""

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "m3s.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(m3s_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available to build the library")
    from nvfp4_block_sparse_m3s_gb300 import binding
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("m3s_nvfp4_store", "m3s_decode_rows", "m3s_index_score_topk",
              "m3s_verify_score_topk", "m3s_sparse_attention", "m3s_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.m3s_version().startswith(b"m3s")


def test_workspace_sizes(lib):
    from nvfp4_block_sparse_m3s_gb300 import binding as M
    # up to 256 tiles (index: a tile per row; verify: up to 8 rows of one request):
    # two launches, the block scores (rows x bt_stride fp32) in the workspace
    assert M.m3s_workspace_bytes(M.OP_INDEX_SCORE_TOPK, 8, 8, 3600, 0, 0, 16, 16) == 8 * 3600 * 4
    assert M.m3s_workspace_bytes(M.OP_VERIFY_SCORE_TOPK, 128, 16, 1600, 0, 0, 16, 16, 8) == \
        128 * 1600 * 4
    # more tiles: the streaming top-k's state, a ticket per tile (256-byte rounded),
    # candidate lists for ntiles + 255 slots of rows-per-tile x topk 8-byte keys and
    # (verify) each CTA's segment score scratch (8 rows x bt_stride fp32)
    assert M.m3s_workspace_bytes(M.OP_INDEX_SCORE_TOPK, 300, 300, 24, 0, 0, 16, 16) == \
        1280 + (300 + 255) * 1 * 16 * 8
    assert M.m3s_workspace_bytes(M.OP_VERIFY_SCORE_TOPK, 8192, 1, 2112, 0, 0, 16, 16, 8192) == \
        4096 + (1024 + 255) * 8 * 16 * 8 + 256 * 8 * 2112 * 4
    assert M.m3s_workspace_bytes(M.OP_INDEX_SCORE_TOPK, 8, 8, 3600, 0, 0, 16, 0) == 0   # no top-k
    # a slice's candidates: always the streaming state, whatever the row count
    assert M.m3s_workspace_bytes(M.OP_INDEX_CANDIDATES, 8, 8, 3600, 0, 0, 16, 16) == \
        256 + (8 + 255) * 1 * 16 * 8
    assert M.m3s_workspace_bytes(M.OP_INDEX_CANDIDATES, 300, 300, 24, 0, 0, 16, 16) == \
        1280 + (300 + 255) * 1 * 16 * 8
    # the two-launch decode step: candidate lists for R + 255 slots (256-byte
    # rounded), then an (first slot, lists) pair a row
    assert M.m3s_workspace_bytes(M.OP_INDEX_ATTENTION, 8, 8, 3600, 16, 1, 16, 16) == \
        (263 * 16 * 8 + 255) // 256 * 256 + 8 * 8
    assert M.m3s_workspace_bytes(M.OP_INDEX_ATTENTION, 8, 8, 3600, 16, 1, 16, 0) == 0
    # the two-launch verify step: lists for (16 tiles + 255) slots of 8 rows, a
    # 256 x 8 x 1500 fp32 block-maximum scratch, an int2 per row (each part
    # 256-byte rounded); 0 past 8192 tiles
    cand = (16 + 255) * 8 * 16 * 8
    seg = 256 * 8 * 1500 * 4
    assert M.m3s_workspace_bytes(M.OP_VERIFY_INDEX_ATTENTION, 128, 16, 1500, 16, 1, 16, 16, 8) == \
        ((cand + 255) // 256 * 256 + seg + 255) // 256 * 256 + 128 * 8
    assert M.m3s_workspace_bytes(M.OP_VERIFY_INDEX_ATTENTION, 128, 16, 1500, 16, 1, 16, 0, 8) == 0
    assert M.m3s_workspace_bytes(M.OP_VERIFY_INDEX_ATTENTION, 128, 8193, 1500, 16, 1, 16, 16, 8) == 0
    assert M.m3s_workspace_bytes(M.OP_VERIFY_SCORE_TOPK, 0, 8, 3600) == 0
    # attention merges its split-K partials on chip (thread-block cluster): no workspace
    assert M.m3s_workspace_bytes(M.OP_SPARSE_ATTENTION, 8, 8, 3600, 16, 1, 16, 16) == 0
    assert M.m3s_workspace_bytes(M.OP_SPARSE_ATTENTION, 8192, 1, 2112, 16, 1, 16, 16) == 0
    assert M.m3s_workspace_bytes(99, 8, 8, 8) == 0
    # more than 8192 tiles: the calls reject the shape first, so there is no size
    # (also no signed overflow for the largest int32 row count)
    for op in (M.OP_INDEX_SCORE_TOPK, M.OP_INDEX_CANDIDATES, M.OP_INDEX_ATTENTION):
        assert M.m3s_workspace_bytes(op, 8192, 8192, 64, 16, 1, 16, 16) > 0
        assert M.m3s_workspace_bytes(op, 8193, 8193, 64, 16, 1, 16, 16) == 0
        assert M.m3s_workspace_bytes(op, 2 ** 31 - 1, 8, 64, 16, 1, 16, 16) == 0
    assert M.m3s_workspace_bytes(M.OP_VERIFY_SCORE_TOPK, 128, 1025, 64, 0, 0, 16, 16, 64) == 0
    assert M.m3s_workspace_bytes(M.OP_VERIFY_SCORE_TOPK, 128, 1024, 64, 0, 0, 16, 16, 64) > 0


def test_host_validation_rejects_before_launch(lib):
    from nvfp4_block_sparse_m3s_gb300 import binding as M
    P = M.Plane(None, None, 4, 1)
    # null source
    assert lib.m3s_nvfp4_store(None, 128, 4, 1, None, P, None, None) == M.ERR_INVALID
    # head count mismatch with the plane
    assert lib.m3s_nvfp4_store(None, 128, 4, 2, None, P, None, None) == M.ERR_INVALID
    # nothing to do
    assert lib.m3s_nvfp4_store(None, 128, 0, 1, None, P, None, None) == M.OK
    assert lib.m3s_decode_rows(None, None, 1, 0, None, None, None) == M.OK
    assert lib.m3s_decode_rows(None, None, -1, 4, None, None, None) == M.ERR_INVALID
    # too many index heads / top-k beyond the build
    assert lib.m3s_index_score_topk(None, None, 17, P, None, 1, None, None, 1, 1, 8, 0, 0, None,
                                    None, None, 0, None, None) == M.ERR_UNSUPPORTED
    assert lib.m3s_index_score_topk(None, None, 16, P, None, 1, None, None, 1, 1, 65, 0, 0, None,
                                    None, None, 0, None, None) == M.ERR_UNSUPPORTED
    # context parallelism: top-k beyond the build, more lists than the merge takes,
    # a slice without its begin / count arrays
    assert lib.m3s_merge_candidates(None, 2, 4, 65, None, None) == M.ERR_UNSUPPORTED
    assert lib.m3s_merge_candidates(None, 257, 4, 16, None, None) == M.ERR_UNSUPPORTED
    assert lib.m3s_merge_candidates(None, 2, 4, 16, None, None) == M.ERR_INVALID
    assert lib.m3s_merge_candidates(None, 2, 0, 16, None, None) == M.OK
    fake_plane = M.Plane(ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21), 4, 1)
    fk = ctypes.c_void_p(1 << 20)
    assert lib.m3s_index_score_candidates(fk, fk, 16, fake_plane, fk, 4, None, None, fk, fk, 2, 2,
                                          16, 0, 0, fk, fk, 1 << 20, None, None) == M.ERR_INVALID
    # the two-launch decode step checks the attention's arguments before it
    # launches anything: q heads not a multiple of KV heads, GQA beyond 16
    fk2 = ctypes.c_void_p(1 << 20)
    P3 = M.Plane(ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21), 4, 1)
    assert lib.m3s_index_attention(fk2, fk2, 16, P3, fk2, 6, 4, P3, P3, fk2, 4, 2, fk2, fk2, 2, 16, 0, 0,
                                   ctypes.c_float(0.1), fk2, fk2, None, fk2, 1 << 20, None, None) == M.ERR_INVALID
    assert lib.m3s_index_attention(fk2, fk2, 16, P3, fk2, 32, 1, P3, P3, fk2, 4, 2, fk2, fk2, 2, 16, 0, 0,
                                   ctypes.c_float(0.1), fk2, fk2, None, fk2, 1 << 20, None,
                                   None) == M.ERR_UNSUPPORTED
    assert lib.m3s_index_attention(fk2, fk2, 16, P3, fk2, 16, 1, P3, P3, fk2, 4, 2, fk2, fk2, 2, 16, 0, 0,
                                   ctypes.c_float(0.1), fk2, fk2, None, fk2, 16, None, None) == M.ERR_WORKSPACE
    # the two-launch verify step: the attention's checks, then cu_q, the tile
    # count and the workspace, before anything is launched
    def via(Hq=16, Hkv=1, cu_q=fk2, B=2, max_q=8, ws_bytes=1 << 30):
        return lib.m3s_verify_index_attention(fk2, fk2, 16, P3, fk2, Hq, Hkv, P3, P3, fk2, 4, B, cu_q, fk2, fk2,
                                              2, max_q, 16, 0, 0, ctypes.c_float(0.1), fk2, fk2, None, fk2,
                                              ws_bytes, None, None)
    assert via(Hq=6, Hkv=4) == M.ERR_INVALID
    assert via(cu_q=None) == M.ERR_INVALID
    assert via(max_q=-1) == M.ERR_INVALID
    assert via(B=8193) == M.ERR_UNSUPPORTED
    assert via(ws_bytes=16) == M.ERR_WORKSPACE
    # the store with the row map: negative counts, a row map without outputs
    assert lib.m3s_nvfp4_store_batch_rows(None, 0, 0, None, None, None, -1, 4, None, None, None,
                                          None) == M.ERR_INVALID
    assert lib.m3s_nvfp4_store_batch_rows(None, 0, 0, None, fk2, fk2, 2, 4, None, None, None,
                                          None) == M.ERR_INVALID
    assert lib.m3s_nvfp4_store_batch_rows(None, 0, 0, None, None, None, 0, 0, None, None, None,
                                          None) == M.OK
    # forced block counts must not be negative
    fake = ctypes.c_void_p(1 << 20)
    assert lib.m3s_block_topk(fake, 8, fake, fake, 1, 1, 8, 4, -1, 0, fake, None) == M.ERR_INVALID
    assert lib.m3s_block_topk(fake, 8, fake, fake, 1, 1, 8, 4, 0, -2, fake, None) == M.ERR_INVALID
    # attention: q heads not a multiple of KV heads, GQA beyond 16
    P2 = M.Plane(None, None, 4, 1)
    assert lib.m3s_sparse_attention(None, 6, 4, P2, P2, None, 1, 1, None, None, None, 16, 1,
                                    ctypes.c_float(0.1), None, None, None, 0, None,
                                    None) == M.ERR_INVALID
    assert lib.m3s_sparse_attention(None, 32, 1, P2, P2, None, 1, 1, None, None, None, 16, 1,
                                    ctypes.c_float(0.1), None, None, None, 0, None,
                                    None) == M.ERR_UNSUPPORTED


def test_plane_format_rules(lib):
    """A plane's format field: 0 = NVFP4, 1 = MXFP4, anything else is rejected; K and V
    must share one format. All decided on the host (the fake device pointers are
    never dereferenced and nothing is launched)."""
    from nvfp4_block_sparse_m3s_gb300 import binding as M
    fake = ctypes.c_void_p(1 << 20)
    nv = M.Plane(fake, fake, 4, 1, M.FMT_NVFP4)
    mx = M.Plane(fake, fake, 4, 1, M.FMT_MXFP4)
    bad = M.Plane(fake, fake, 4, 1, 7)
    assert ctypes.sizeof(M.Plane) == 32
    # store: an unknown format is an invalid argument
    assert lib.m3s_nvfp4_store(fake, 128, 4, 1, fake, bad, None, None) == M.ERR_INVALID
    # index scorer: unknown format rejected; both known formats pass validation (checked
    # with R = 0, which returns before any launch)
    assert lib.m3s_index_score_topk(fake, fake, 16, bad, fake, 8, fake, fake, 1, 1, 8, 0, 0, fake,
                                    None, fake, 1 << 20, None, None) == M.ERR_INVALID
    for p in (nv, mx):
        assert lib.m3s_index_score_topk(fake, fake, 16, p, fake, 8, fake, fake, 0, 1, 8, 0, 0, fake,
                                        None, fake, 1 << 20, None, None) == M.OK
    # fused verify: both formats pass validation (R = 0: nothing is launched), an
    # unknown one is rejected before any launch
    for p in (nv, mx):
        assert lib.m3s_verify_score_topk(fake, fake, 16, p, fake, 8, fake, fake, 1, 0, 8, 16, 0, 0,
                                         fake, fake, 1 << 20, None, None) == M.OK
    assert lib.m3s_verify_score_topk(fake, fake, 16, bad, fake, 8, fake, fake, 1, 1, 8, 16, 0, 0,
                                     fake, fake, 1 << 20, None, None) == M.ERR_INVALID
    # attention: mixed K / V formats refused, unknown format invalid
    args = (fake, 1, 1, fake, fake, fake, 16, 1, ctypes.c_float(0.1), fake, None, None, 0, None, None)
    assert lib.m3s_sparse_attention(fake, 16, 1, nv, mx, *args) == M.ERR_UNSUPPORTED
    assert lib.m3s_sparse_attention(fake, 16, 1, bad, bad, *args) == M.ERR_INVALID


def test_quantise_at_write_host_validation(lib):
    """m3s_qk_norm_rope_store rejects bad jobs and rotary sizes on the host (nothing
    is launched: every call below either fails validation or has T = 0)."""
    from nvfp4_block_sparse_m3s_gb300 import binding as M
    fake = ctypes.c_void_p(1 << 20)
    plane = M.Plane(fake, fake, 4, 2, M.FMT_NVFP4)

    def job(H=2, stride=256, weight=None, rope=0, dst=plane, out=None, out_stride=0):
        return M.WriteJob(fake, stride, H, weight, rope, dst, out, out_stride)

    def call(jobs, T=1, cos=fake, sin=fake, rd=64, slots=fake):
        arr = (M.WriteJob * len(jobs))(*jobs)
        return lib.m3s_qk_norm_rope_store(arr, len(jobs), T, slots, cos, sin, rd,
                                          ctypes.c_float(1e-6), None, None)
    assert call([job(rope=1)], rd=60) == M.ERR_INVALID           # not a multiple of 8
    assert call([job(rope=1)], rd=136) == M.ERR_INVALID          # beyond head_dim
    assert call([job(rope=1)], cos=None) == M.ERR_INVALID        # no table
    assert call([job(stride=100)]) == M.ERR_INVALID              # row stride below H * 128
    assert call([job(H=3)]) == M.ERR_INVALID                     # plane heads mismatch
    assert call([job(dst=M.Plane(fake, fake, 4, 2, 5))]) == M.ERR_INVALID   # unknown format
    assert call([job(out=fake, out_stride=200)]) == M.ERR_INVALID          # short output rows
    assert call([job()], slots=None) == M.ERR_INVALID           # plane job without slots
    assert call([job()] * 7) == M.ERR_INVALID                    # too many jobs
    assert call([job(rope=1), job(out=fake, out_stride=256)], T=0) == M.OK


def test_binding_checks_raise_type_errors_on_host_tensors():
    """The binding's argument checks are explicit TypeErrors (they hold under
    python -O): plane layouts, store rows. Host tensors suffice: nothing is
    launched before the checks."""
    import torch
    from nvfp4_block_sparse_m3s_gb300 import binding as M
    codes = torch.zeros((4, 1, 128, 64), dtype=torch.uint8)
    nv = torch.zeros((4, 1, 128, 8), dtype=torch.uint8)
    mx = torch.zeros((4, 1, 128, 4), dtype=torch.uint8)
    assert M.plane(codes, nv).format == M.FMT_NVFP4
    assert M.plane(codes, mx).format == M.FMT_MXFP4
    p = M.plane(codes, nv)
    assert (p.num_pages, p.num_heads) == (4, 1)
    for bad in ((codes.float(), nv), (codes, nv.float()), (codes[:, :, :, :32], nv), (codes, nv[:2]),
                (codes, torch.zeros((4, 1, 128, 6), dtype=torch.uint8)), (codes.transpose(0, 1), nv),
                (codes[..., ::2], nv)):
        with pytest.raises(TypeError):
            M.plane(*bad)
    rows = torch.zeros((5, 1, 128), dtype=torch.bfloat16)
    M._store_job(rows, 5, codes, nv)
    for bad_rows, T in ((rows.float(), 5), (rows, 4), (rows[:, :, :64], 5),
                        (torch.zeros((5, 2, 256), dtype=torch.bfloat16)[:, :, :128], 5)):
        with pytest.raises(TypeError):
            M._store_job(bad_rows, T, codes, nv)


def test_header_is_plain_c_and_the_library_links_from_c(lib, tmp_path):
    """A C11 host program (gcc -pedantic -Werror, no C++) that takes the address
    of every declared function links against libm3s.so, and on a machine
    without a GPU its host-only calls work: the version, a workspace size
    (equal to the ctypes binding's) and an argument check answered before any
    launch."""
    import subprocess

    from nvfp4_block_sparse_m3s_gb300 import binding as M
    from nvfp4_block_sparse_m3s_gb300 import build as B
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    names = declared_functions()
    prog = "\n".join([
        "#include <stdio.h>",
        '#include "m3s.h"',
        "typedef void (*fn_t)(void);",
        "static fn_t all_fns[] = {" + ", ".join(f"(fn_t){n}" for n in names) + "};",
        "int main(void) {",
        "  m3s_fp4_plane p = {NULL, NULL, 4, 4, M3S_FMT_NVFP4};",
        "  size_t ws = m3s_workspace_bytes(M3S_OP_INDEX_ATTENTION, 8, 8, 4096, 16, 1, 16, 16, 1);",
        "  int rc = m3s_sparse_attention(NULL, 6, 4, p, p, NULL, 1, 1, NULL, NULL, NULL, 16, 1, 0.1f,",
        "                                NULL, NULL, NULL, 0, NULL, NULL);",
        '  printf("%s|%zu|%d|%d\\n", m3s_version(), ws, rc, (int)(sizeof(all_fns) / sizeof(all_fns[0])));',
        "  return 0;",
        "}",
    ])
    src = tmp_path / "host.c"
    src.write_text(prog)
    exe = tmp_path / "host"
    libdir = os.path.dirname(B.LIB)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", libdir, "-lm3s", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.strip().split("|")
    assert out[0] == lib.m3s_version().decode()
    assert int(out[1]) == M.m3s_workspace_bytes(M.OP_INDEX_ATTENTION, 8, 8, 4096, 16, 1, 16, 16, 1) > 0
    assert int(out[2]) == M.ERR_INVALID
    assert int(out[3]) == len(names)


def test_binding_signatures_match_the_header():
    """The ctypes binding declares every header function, with as many
    parameters as the declaration (an undeclared one would pass 64-bit
    pointers as C int; a count that drifted would shift the arguments)."""
    from nvfp4_block_sparse_m3s_gb300 import binding as M
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = dict(re.findall(r"\b(m3s_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text))
    assert set(decls) == set(declared_functions()) == set(M._SIGS)
    for name, params in decls.items():
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(M._SIGS[name][1]) == n, (name, n, len(M._SIGS[name][1]))
