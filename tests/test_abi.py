"""The C ABI without a GPU: the library loads, exports every declared symbol, the ctypes structs
match the C layout, and host-side validation returns the documented codes (no kernel runs)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specdec.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|void|const char\s*\*)\s+(specdec_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported():
    import speculative_decoding_specdec_gb300.specdec as sd
    names = declared_functions()
    assert "specdec_realign" in names and "specdec_verify_sample" in names
    assert "specdec_verify_greedy_workspace" in names and "specdec_verify_greedy_noalloc" in names
    assert "specdec_pool_schedule" in names and "specdec_arena_destroy" in names
    assert "specdec_verify_sample_philox" in names and "specdec_philox_uniforms" in names
    missing = [n for n in names if not hasattr(sd.lib, n)]
    assert missing == []
    assert sd.version() == 100


def test_header_constants_match_binding():
    import speculative_decoding_specdec_gb300.specdec as sd
    text = open(HEADER).read()
    macro = {m: int(v) for m, v in re.findall(r"^#define (SPECDEC_\w+) (\d+)", text, re.M)}
    assert macro["SPECDEC_MAX_DRAFT"] == sd.MAX_DRAFT
    assert macro["SPECDEC_GREEDY_SCRATCH_BYTES"] == sd.GREEDY_SCRATCH_BYTES
    assert macro["SPECDEC_REALIGN_PDL"] == sd.REALIGN_PDL


def test_status_strings():
    import speculative_decoding_specdec_gb300.specdec as sd
    assert sd.status_string(0) == "ok"
    assert "capacity" in sd.status_string(4)
    assert sd.status_string(99) == "unknown status"


STRUCT_PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "specdec.h"
#define F(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("specdec_kv_view %zu\n", sizeof(specdec_kv_view));
  printf("specdec_realign_args %zu\n", sizeof(specdec_realign_args));
  printf("specdec_pool_args %zu\n", sizeof(specdec_pool_args));
  printf("specdec_keep_bound %zu\n", sizeof(specdec_keep_bound));
  printf("specdec_schedule_args %zu\n", sizeof(specdec_schedule_args));
  printf("specdec_admit_args %zu\n", sizeof(specdec_admit_args));
  %FIELDS%
  return 0;
}
"""


def test_ctypes_layout_matches_c(tmp_path):
    import speculative_decoding_specdec_gb300.specdec as sd
    structs = {"specdec_kv_view": sd.KvView, "specdec_realign_args": sd.RealignArgs,
               "specdec_pool_args": sd.PoolArgs, "specdec_keep_bound": sd.KeepBound,
               "specdec_schedule_args": sd.ScheduleArgs, "specdec_admit_args": sd.AdmitArgs}
    fields = "\n".join(f"F({cn}, {f})" for cn, py in structs.items() for f, _ in py._fields_)
    src = tmp_path / "probe.c"
    src.write_text(STRUCT_PROBE.replace("%FIELDS%", fields))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    out = dict(line.rsplit(" ", 1) for line in
               subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
               if line)
    for cn, py in structs.items():
        assert int(out[cn]) == ctypes.sizeof(py), cn
        for f, _ in py._fields_:
            assert int(out[f"{cn}.{f}"]) == getattr(py, f).offset, (cn, f)


def test_host_validation_codes():
    import speculative_decoding_specdec_gb300.specdec as sd
    L = sd.lib
    # verify_greedy: empty batch is a no-op; bad sizes and NULL pointers are caught on the host
    assert L.specdec_verify_greedy(None, sd.BF16, 0, 4, 100, 100, None, None, None, None, 0, None, None) == sd.OK
    assert L.specdec_verify_greedy(None, sd.BF16, 1, 4, 100, 100, None, None, None, None, 0, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy(None, sd.BF16, 1, 0, 100, 100, None, None, None, None, 0, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy(None, sd.BF16, 1, 32, 100, 100, None, None, None, None, 0, None, None) == sd.ERR_UNSUPPORTED
    assert L.specdec_verify_greedy(None, 7, 1, 4, 100, 100, None, None, None, None, 0, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy(None, sd.F32, 1, 4, 100, 99, None, None, None, None, 0, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy_workspace(0, 4) == 0                        # invalid shape
    # the workspace-free variant applies the same host checks before it touches a device
    assert L.specdec_verify_greedy_noalloc(None, sd.BF16, 0, 4, 100, 100, None, None, None, None, None) == sd.OK
    assert L.specdec_verify_greedy_noalloc(None, sd.BF16, 1, 0, 100, 100, None, None, None, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy_noalloc(None, sd.BF16, 1, 32, 100, 100, None, None, None, None, None) == sd.ERR_UNSUPPORTED
    # a shape beyond the static scratch: argument mistakes are reported as by the workspace entry
    # point first (NULL pointers, bad dtype, row stride below V), then the scratch limit
    assert L.specdec_verify_greedy_noalloc(None, sd.BF16, 4096, 5, 100, 100, None, None, None, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy_noalloc(None, 7, 4096, 5, 100, 100, None, None, None, None, None) == sd.ERR_INVALID_ARG
    fake = 1 << 20        # stand-in device addresses: the host checks never dereference them
    assert L.specdec_verify_greedy_noalloc(fake, sd.BF16, 4096, 5, 100, 99, fake, fake, fake, fake, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy_noalloc(fake + 1, sd.BF16, 4096, 5, 100, 100, fake, fake, fake, fake, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy_noalloc(fake, sd.BF16, 4096, 5, 100, 100, fake, fake, fake, fake, None) == sd.ERR_UNSUPPORTED
    # the wait self-test checks its limits on the host
    assert L.specdec_wait_selftest(0, 0, 1 << 20, None) == sd.ERR_INVALID_ARG
    assert L.specdec_wait_selftest(1, 0, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_wait_selftest(1, 2000000, 1 << 20, None) == sd.ERR_INVALID_ARG
    assert L.specdec_verify_greedy_workspace(3, 32) == 0
    assert L.specdec_verify_greedy_workspace(3, 4) == 256 + 256               # keys, counters
    # realign: NULL args, empty batch, bad views
    assert L.specdec_realign(None, None) == sd.ERR_INVALID_ARG
    a = sd.RealignArgs()
    a.B, a.D = 0, 4
    assert L.specdec_realign(ctypes.byref(a), None) == sd.OK
    a.B = 2
    assert L.specdec_realign(ctypes.byref(a), None) == sd.ERR_INVALID_ARG     # NULL cache base
    a.src = sd.KvView(16, 64, 32, 16, 8, sd.BF16, 1, 2, 1, 4, 2)            # head_dim*2 = 8 bytes
    a.dst = sd.KvView(4096, 64, 32, 16, 8, sd.BF16, 1, 2, 1, 4, 2)
    assert L.specdec_realign(ctypes.byref(a), None) == sd.ERR_UNSUPPORTED
    a.D = 40
    assert L.specdec_realign(ctypes.byref(a), None) == sd.ERR_UNSUPPORTED
    # in place: the destination must be the source view (checked before any pointer is used)
    a.D = 4
    a.src = sd.KvView(4096, 64, 32, 16, 8, sd.BF16, 1, 2, 1, 8, 2)             # 16-byte columns
    a.dst = sd.KvView(8192, 64, 32, 16, 8, sd.BF16, 1, 2, 1, 8, 2)
    assert L.specdec_realign_inplace(ctypes.byref(a), None) == sd.ERR_INVALID_ARG
    assert L.specdec_realign_inplace(None, None) == sd.ERR_INVALID_ARG
    a.flags = 2                                                              # unknown flag
    assert L.specdec_realign(ctypes.byref(a), None) == sd.ERR_INVALID_ARG
    a.flags = 0
    a.schedule = 4098                                        # scheduling words not 4-byte aligned
    assert L.specdec_realign(ctypes.byref(a), None) == sd.ERR_INVALID_ARG
    assert L.specdec_realign_inplace(ctypes.byref(a), None) == sd.ERR_INVALID_ARG
    a.B = 0
    assert L.specdec_realign(ctypes.byref(a), None) == sd.ERR_INVALID_ARG
    a.schedule, a.B = None, 2
    # grouping
    assert L.specdec_group_by_length(None, -1, 8, 10, None, None, None, None, None, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_group_by_length(None, 5000, 8, 10, None, None, None, None, None, None, None) == sd.ERR_UNSUPPORTED
    assert L.specdec_group_by_length(None, 4, 8, 20000, None, None, None, None, None, None, None) == sd.ERR_UNSUPPORTED
    assert L.specdec_group_by_length(None, 4, 0, 10, None, None, None, None, None, None, None) == sd.ERR_INVALID_ARG
    # pool moves
    assert L.specdec_pool_gather(None, None) == sd.ERR_INVALID_ARG
    p = sd.PoolArgs()
    assert L.specdec_pool_append(ctypes.byref(p), None) == sd.ERR_INVALID_ARG
    # in-kernel uniforms
    assert L.specdec_philox_uniforms(1, 2, 0, 3, None, None) == sd.OK                  # nothing to draw
    assert L.specdec_philox_uniforms(1, 2, 4, 3, None, None) == sd.ERR_INVALID_ARG     # NULL out
    assert L.specdec_philox_uniforms(1, 2, 4, 0, None, None) == sd.ERR_INVALID_ARG
    assert L.specdec_philox_uniforms(1, 2, 4, 32, None, None) == sd.ERR_UNSUPPORTED
    assert L.specdec_verify_sample_philox(None, None, sd.BF16, 0, 4, 100, 100, 1.0, None, 1, 2,
                                          None, None, None, None, None, None) == sd.OK
    assert L.specdec_verify_sample_philox(None, None, sd.BF16, 2, 4, 100, 100, 1.0, None, 1, 2,
                                          None, None, None, None, None, None) == sd.ERR_INVALID_ARG
    # lifecycle: schedule and admission (host checks; no kernel runs)
    assert L.specdec_pool_schedule(None, None) == sd.ERR_INVALID_ARG
    g = sd.ScheduleArgs()
    g.S, g.batch_size, g.window = 4, 0, 0
    assert L.specdec_pool_schedule(ctypes.byref(g), None) == sd.ERR_INVALID_ARG   # batch size 0
    g.batch_size, g.window = 8, -1
    assert L.specdec_pool_schedule(ctypes.byref(g), None) == sd.ERR_INVALID_ARG   # negative window
    g.S, g.window = 5000, 0
    assert L.specdec_pool_schedule(ctypes.byref(g), None) == sd.ERR_UNSUPPORTED   # > 4096 slots
    g.S = 4
    assert L.specdec_pool_schedule(ctypes.byref(g), None) == sd.ERR_INVALID_ARG   # NULL buffers
    m = sd.AdmitArgs()
    m.n, m.S, m.D, m.ids_cap = 0, 4, 3, 16
    assert L.specdec_pool_admit(ctypes.byref(m), None) == sd.OK                   # nothing to admit
    m.n = 2
    assert L.specdec_pool_admit(ctypes.byref(m), None) == sd.ERR_INVALID_ARG      # NULL buffers
    m.n = 2000
    assert L.specdec_pool_admit(ctypes.byref(m), None) == sd.ERR_UNSUPPORTED      # > 1024 entries
    m.n, m.D = 2, 0
    assert L.specdec_pool_admit(ctypes.byref(m), None) == sd.ERR_INVALID_ARG
    assert L.specdec_pool_admit(None, None) == sd.ERR_INVALID_ARG
    # retirement needs the limits
    p.slot_state = 64
    assert L.specdec_pool_append(ctypes.byref(p), None) == sd.ERR_INVALID_ARG


def test_arena_allocator_matches_first_fit_oracle():
    """The host allocator (C++) against the oracle's bitmap first fit: same columns for the same
    sequence of requests and frees, same free totals."""
    import numpy as np
    import speculative_decoding_specdec_gb300.specdec as sd
    import oracle.specdec_oracle as O
    rng = np.random.default_rng(5)
    for cols in (1, 17, 500):
        a, o = sd.Arena(cols), O.FirstFitArena(cols)
        live = []
        for _ in range(400):
            if live and rng.random() < 0.45:
                c = live.pop(int(rng.integers(len(live))))
                a.free(c)
                o.free(c)
            else:
                n = int(rng.integers(1, max(2, cols // 4)))
                got = a.alloc(n)
                try:
                    want = o.alloc(n)
                except O.OracleError:
                    want = None
                assert got == want
                if got is not None:
                    live.append(got)
            assert a.stats() == (o.free_cols(), o.largest_free(), len(live))
        with pytest.raises(sd.SpecdecError):
            a.free(cols + 5)                                       # not an allocation
        with pytest.raises(sd.SpecdecError):
            a.alloc(0)                                             # empty request
        for c in live:
            a.free(c)
        assert a.stats() == (cols, cols, 0) and a.alloc(cols) == 0


def test_binding_raises_on_host_error():
    import speculative_decoding_specdec_gb300.specdec as sd
    with pytest.raises(sd.SpecdecError) as e:
        sd._check(sd.ERR_CAPACITY, "x")
    assert e.value.code == sd.ERR_CAPACITY
