"""The C ABI without a GPU: libpg.so builds, loads, exports every function that
include/pg.h declares, and its host-side checks answer before any CUDA work."""
import ctypes
import os
import re
import subprocess

import pytest

from hashed_head_gram_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pg.h")


@pytest.fixture(scope="module")
def pg():
    from hashed_head_gram_gb300.build import build
    build()
    from hashed_head_gram_gb300 import pg as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_lookup_calls():
    names = declared_functions()
    for n in ("pg_canon_hash", "pg_gather_sign_concat", "pg_project_gate", "pg_conv_residual"):
        assert n in names


def test_library_exports_every_declared_function(pg):
    lib_path = os.path.join(ROOT, "hashed_head_gram_gb300", "libpg.so")
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pg_[a-z0-9_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(pg.lib(), n) is not None


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "pg.h"\nint main(void){pg_table_desc d; (void)d; return (int)sizeof(d) > 0 ? 0 : 1;}\n')
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I" + os.path.join(ROOT, "include"),
                           "-c", str(src), "-o", str(tmp_path / "t.o")])


def test_descriptor_layout_matches_the_header(pg, tmp_path):
    src = tmp_path / "sz.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "pg.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu\\n", sizeof(pg_table_desc),'
                   ' offsetof(pg_table_desc, hash_seed), offsetof(pg_table_desc, rows),'
                   ' offsetof(pg_table_desc, canon_vocab)); return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.check_call(["gcc", "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    size, seed_off, rows_off, cv_off = map(int, subprocess.check_output([str(exe)]).split())
    T = pg.TableDesc
    assert ctypes.sizeof(T) == size and T.hash_seed.offset == seed_off
    assert T.rows.offset == rows_off and T.canon_vocab.offset == cv_off


def test_status_strings_and_version(pg):
    L = pg.lib()
    assert L.pg_abi_version() == 1
    for s in range(11):
        assert L.pg_status_str(s)
    assert L.pg_status_str(99) == b"unknown status"


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_geometry_of_every_workload(pg, cfg):
    w = W.make_workload(cfg)
    for spec in w.tables:
        rows, rb, ew = pg.table_geometry(pg.table_desc(spec, w.vocab, w.canon_vocab))
        assert (rows, rb, ew) == (spec.table_rows, spec.row_bytes, spec.e_width)


def test_descriptor_validation(pg):
    spec = W.make_workload(2).tables[0]
    cases = []
    d = pg.table_desc(spec, 50304); d.abi_version = 9; cases.append((d, 7))
    d = pg.table_desc(spec, 50304); d.orders[1] = 2; cases.append((d, 2))           # not increasing
    d = pg.table_desc(spec, 50304); d.K = 17; cases.append((d, 2))
    d = pg.table_desc(spec, 50304); d.pages[0] = 0; cases.append((d, 2))
    d = pg.table_desc(spec, 50304); d.row_dtype = 7; cases.append((d, 3))
    d = pg.table_desc(spec, 50304); d.row_dtype = 2; d.r = 80; cases.append((d, 3))  # NF4 needs r = 64
    d = pg.table_desc(spec, 50304); d.pages[0] = 0xFFFFFFF; cases.append((d, 4))     # >= 2^32 rows
    d = pg.table_desc(spec, 50304); d.vocab = 0; cases.append((d, 2))
    for desc, want in cases:
        with pytest.raises(pg.PgError) as ex:
            pg.table_geometry(desc)
        assert ex.value.status == want


def test_calls_reject_null_pointers_on_the_host(pg):
    L = pg.lib()
    spec = W.make_workload(2).tables[0]
    d = pg.table_desc(spec, 50304)
    assert L.pg_gather_sign_concat(ctypes.byref(d), None, 2, 3, None, None, 0, None, 1, None, None) == 1
    assert L.pg_canon_hash(ctypes.byref(d), None, 2, 3, None, None, None, None, None, None) == 1
    assert L.pg_canon_hash(ctypes.byref(d), None, -1, 3, None, None, None, None, None, None) == 2
    assert L.pg_project_gate(4, 64, 128, 0, 1, None, None, 0, 0.0, None, None, None, None, 1e-6, None, None,
                             None, None, 0, None) == 1
    assert L.pg_project_gate(4, 64, 128, 1, 1, None, None, 0, 0.0, None, None, None, None, 1e-6, None, None,
                             None, None, 0, None) == 2                             # M with gate NONE
    assert L.pg_conv_residual(1, 4, 12, 1, 1, None, None, None, None, None, 4, 3, 1e-6, None, None) == 2  # d % 8
    assert L.pg_conv_residual(1, 4, 16, 1, 1, None, None, None, None, None, 4, 3, 1e-6, None, None) == 1


def test_workspace_size_query(pg):
    # per (branch, 256-column tile) partial sums, + the v tiles' row sums that v_ms_out needs
    assert pg.workspace_size(32768, 1280, 2560, 4, pg.BF16, pg.GATE_CONTEXT) == (4 * 10 * 3 + 10) * 32768 * 4
    assert pg.workspace_size(65536, 1024, 768, 0, pg.BF16, pg.GATE_SCALAR) == 0
    # up to 4 rows (decode batches): the few-rows kernel's 64-column tile sums
    assert pg.workspace_size(4, 1280, 2560, 4, pg.BF16, pg.GATE_CONTEXT) == (4 * 40 * 3 + 40) * 4 * 4
    assert pg.workspace_size(5, 1280, 2560, 4, pg.BF16, pg.GATE_CONTEXT) == (4 * 10 * 3 + 10) * 5 * 4


def test_decode_state_layout_matches_the_header(pg, tmp_path):
    src = tmp_path / "ds.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "pg.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu\\n", sizeof(pg_decode_state),'
                   ' offsetof(pg_decode_state, pos), offsetof(pg_decode_state, ring_v),'
                   ' offsetof(pg_decode_state, ring_ms)); return 0;}\n')
    exe = tmp_path / "ds"
    subprocess.check_call(["gcc", "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    size, pos_off, rv_off, rms_off = map(int, subprocess.check_output([str(exe)]).split())
    T = pg.DecodeStateC
    assert ctypes.sizeof(T) == size and T.pos.offset == pos_off
    assert T.ring_v.offset == rv_off and T.ring_ms.offset == rms_off


def test_decode_state_size_arithmetic(pg):
    # parts pos [B] i32, ids [B][4] u32, ring_v [B][R][d], ring_alpha [B][R][M] f32,
    # ring_ms [B][R] f32, each rounded up to 256 bytes; R = (kernel - 1) * dilation + 1
    up = lambda x: (x + 255) // 256 * 256
    assert pg.decode_state_size(5) == up(20) + up(80)                      # lookup only
    B, d, M, R = 3, 2560, 4, 10                                             # Engram-27B module
    assert pg.decode_state_size(B, d, M, pg.BF16, 4, 3) == (
        up(4 * B) + up(16 * B) + up(B * R * d * 2) + up(B * R * M * 4) + up(B * R * 4))
    assert pg.decode_state_size(2, 64, 1, pg.F32, 4, 8) == up(8) + up(32) + up(2 * 25 * 64 * 4) + up(2 * 25 * 4) * 2
    assert pg.decode_state_size(2, 64, 1, pg.F32, 1, 3) == up(8) + up(32)   # kernel 1: no ring


def test_decode_state_validation(pg):
    L = pg.lib()
    n = ctypes.c_uint64()
    assert L.pg_decode_state_size(0, 0, 0, pg.BF16, 4, 3, ctypes.byref(n)) == 2      # B < 1
    assert L.pg_decode_state_size(2, 12, 1, pg.BF16, 4, 3, ctypes.byref(n)) == 2     # d % 8
    assert L.pg_decode_state_size(2, 16, 0, pg.BF16, 4, 3, ctypes.byref(n)) == 2     # d without M
    assert L.pg_decode_state_size(2, 16, 9, pg.BF16, 4, 3, ctypes.byref(n)) == 2     # M > 8
    assert L.pg_decode_state_size(2, 16, 1, pg.NF4, 4, 3, ctypes.byref(n)) == 3      # dtype
    assert L.pg_decode_state_size(2, 16, 1, pg.BF16, 5, 3, ctypes.byref(n)) == 2     # kernel > 4
    assert L.pg_decode_state_size(2, 16, 1, pg.BF16, 4, 9, ctypes.byref(n)) == 2     # dilation > 8
    assert L.pg_decode_state_size(2, 16, 1, pg.BF16, 4, 3, None) == 1
    assert L.pg_decode_state_init(None, None, 0, 2, 0, 0, pg.BF16, 4, 3, None) == 1
    st = pg.DecodeStateC()
    assert L.pg_decode_state_init(ctypes.byref(st), ctypes.c_void_p(256), 16, 2, 0, 0, pg.BF16, 4, 3, None) == 8
    assert L.pg_decode_state_init(ctypes.byref(st), ctypes.c_void_p(260), 4096, 2, 0, 0, pg.BF16, 4, 3, None) == 5
    # calls check the state before anything else: missing parts, a conv call on a
    # lookup-only state, a ring depth that disagrees with the conv
    spec = W.make_workload(2).tables[0]
    d = pg.table_desc(spec, 50304)
    st = pg.DecodeStateC(B=2, d=0, M=0, dtype=pg.BF16, kernel_size=4, dilation=3, depth=0)
    assert L.pg_decode_lookup(ctypes.byref(d), ctypes.byref(st), None, None, None, 0, None, 1, None, None) == 1
    st.pos, st.ids = 256, 512
    assert L.pg_decode_conv_residual(ctypes.byref(st), None, None, None, None, None, 1e-6, None, None) == 2
    st = pg.DecodeStateC(B=2, d=64, M=1, dtype=pg.BF16, kernel_size=4, dilation=3, depth=9, pos=256, ids=512)
    assert L.pg_decode_conv_residual(ctypes.byref(st), None, None, None, None, None, 1e-6, None, None) == 2
    st.depth = 10
    assert L.pg_decode_conv_residual(ctypes.byref(st), None, None, None, None, None, 1e-6, None, None) == 1
    ok = pg.DecodeStateC(B=2, d=0, M=0, dtype=pg.BF16, kernel_size=4, dilation=3, depth=0, pos=256, ids=512)
    assert L.pg_decode_reset(ctypes.byref(ok), None, -1, None) == 2
    assert L.pg_decode_reset(ctypes.byref(ok), None, 0, None) == 0
    assert L.pg_decode_reset(ctypes.byref(ok), None, 3, None) == 1


def test_collision_counts_host_checks(pg):
    L = pg.lib()
    b = ctypes.c_size_t()
    assert L.pg_collision_counts_workspace_size(10, 0, ctypes.byref(b)) == 2          # empty span
    assert L.pg_collision_counts_workspace_size(-1, 5, ctypes.byref(b)) == 2
    assert L.pg_collision_counts_workspace_size(10, 5000, None) == 1
    assert L.pg_collision_counts_workspace_size(10, 5000, ctypes.byref(b)) == 0
    assert b.value >= 4 * (5000 + 5001 + 10)                                         # cursors, offsets, indices
    assert L.pg_collision_counts(None, 10, 0, 8, 0, 100, None, None, 0, None) == 2      # K < 1
    assert L.pg_collision_counts(None, 10, 17, 17, 0, 100, None, None, 0, None) == 2    # K > 16
    assert L.pg_collision_counts(None, 10, 8, 4, 0, 100, None, None, 0, None) == 2      # stride < K
    assert L.pg_collision_counts(None, 10, 8, 8, 0, 100, None, None, 0, None) == 1      # no counts
    assert L.pg_collision_counts(None, 10, 8, 8, 0, 100, ctypes.c_void_p(4), None, 0, None) == 5
    assert L.pg_collision_counts(None, 10, 8, 8, 0, 100, ctypes.c_void_p(8), None, 0, None) == 1


def test_row_copy_window_and_host_checks(pg):
    # the window: the 16-byte chunks that hold a row wherever a row of that size can start
    for rb, wb in ((128, 128), (160, 160), (16, 16), (34, 48), (2, 16), (3, 32), (24, 32), (4096, 4096)):
        assert pg.row_copy_window(rb) == wb, rb
    L = pg.lib()
    w = ctypes.c_uint32()
    assert L.pg_row_copy_window(0, ctypes.byref(w)) == 2 and L.pg_row_copy_window(4097, ctypes.byref(w)) == 2
    assert L.pg_row_copy(None, 0, 128, None, 0, None, 0, None) == 0                 # n = 0: nothing to do
    assert L.pg_row_copy(None, 1 << 20, 128, None, 10, None, 0, None) == 1           # PG_ERR_NULL
    assert L.pg_row_copy(None, 1 << 20, 128, None, -1, None, 0, None) == 2           # PG_ERR_SHAPE
    assert L.pg_row_copy(None, 1 << 20, 128, None, 1 << 28, None, 0, None) == 2      # n * 8 chunks >= 2^31
    assert L.pg_row_copy(None, 1 << 20, 34, None, 10, None, 32, None) == 2           # output row < window (48)
    assert L.pg_row_copy(None, 1 << 20, 34, None, 10, None, 136, None) == 2          # not a multiple of 16
    assert L.pg_row_copy(None, 1 << 20, 34, None, 10, None, 128, None) == 1          # valid sizes, NULL pointers


def test_a_c_program_uses_the_library_through_the_header(pg, tmp_path):
    # the boundary is plain C: a C99 program that includes pg.h and links libpg.so runs the
    # host-side calls (no GPU needed for these)
    src = tmp_path / "use_pg.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "pg.h"
int main(void) {
  pg_table_desc d;
  memset(&d, 0, sizeof d);
  d.abi_version = PG_ABI_VERSION; d.hash_version = PG_HASH_VERSION;
  d.mode = PG_PAGEGRAM; d.hash_kind = PG_HASH_MULXOR;
  d.num_orders = 2; d.orders[0] = 2; d.orders[1] = 3;
  d.K = 8; d.S = 4; d.r = 64; d.pages[0] = 48823; d.pages[1] = 48821;
  d.row_dtype = PG_BF16; d.vocab = 50304; d.canon_vocab = 50304;
  uint64_t rows = 0; uint32_t rb = 0, ew = 0;
  pg_status st = pg_table_geometry(&d, &rows, &rb, &ew);
  uint64_t state_bytes = 0;
  pg_status st2 = pg_decode_state_size(64, 2560, 4, PG_BF16, 4, 3, &state_bytes);
  pg_status st3 = pg_gather_sign_concat(&d, NULL, 2, 3, NULL, NULL, 0, NULL, PG_BF16, NULL, NULL);
  printf("%d %llu %u %u %d %llu %d %s\n", (int)st, (unsigned long long)rows, rb, ew, (int)st2,
         (unsigned long long)state_bytes, (int)st3, pg_status_str(PG_ERR_NULL));
  return 0;
}
""")
    lib_dir = os.path.join(ROOT, "hashed_head_gram_gb300")
    exe = tmp_path / "use_pg"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I" + os.path.join(ROOT, "include"), str(src),
                           "-L" + lib_dir, "-l:libpg.so", "-Wl,-rpath," + lib_dir, "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split(maxsplit=7)
    assert out[0] == "0" and int(out[1]) == (48823 + 48821) * 8 * 4 and out[2] == "128" and out[3] == "1024"
    assert out[4] == "0" and int(out[5]) == pg.decode_state_size(64, 2560, 4, pg.BF16, 4, 3)
    assert out[6] == "1" and out[7].strip() == pg.lib().pg_status_str(1).decode()
