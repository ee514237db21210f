"""CPU: the build's register-count gate, the CUDA-core kernel's spill check, and the host-side refusal of a
non-positive bf16/f16 scale."""

import os

import pytest

from paged_kv_cache_181_gb300 import build as b

LOG_OK = """ptxas info    : Compiling entry function '_ZN3foo14attn_tc_kernelILi128ELb1EEEv' for 'sm_103a'
ptxas info    : Function properties for _ZN3foo14attn_tc_kernelILi128ELb1EEEv
    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads
ptxas info    : Used 168 registers, used 16 barriers, 24 bytes cumulative stack size
ptxas info    : Compiling entry function '_ZN3foo10other_kernelEv' for 'sm_103a'
ptxas info    : Used 40 registers, used 0 barriers
ptxas info    : Compiling entry function '_ZN3foo14attn_tc_kernelILi64ELb0EEEv' for 'sm_103a'
ptxas info    : Used 168 registers, used 16 barriers
"""


def test_register_gate_accepts_the_sized_count():
    assert b.check_tc_registers(LOG_OK, 168) == 2


def test_register_gate_refuses_another_count():
    bad = LOG_OK.replace("Used 168 registers, used 16 barriers\n", "Used 170 registers, used 16 barriers\n")
    with pytest.raises(RuntimeError, match="170 registers"):
        b.check_tc_registers(bad, 168)


def test_register_gate_needs_a_report():
    with pytest.raises(RuntimeError, match="no register report"):
        b.check_tc_registers("ptxas info    : Compiling entry function 'x' for 'sm_103a'\n", 168)


def test_register_gate_reads_the_sized_count_from_the_source():
    with open(os.path.join(b.CSRC, b.TC_SOURCE)) as f:
        n = b.expected_tc_registers(f.read())
    assert n == 168
    # The library built in this tree passed the gate: its ptxas report is on disk and agrees.
    log = os.path.join(b.OUT_DIR, b.TC_SOURCE + ".ptxas.txt")
    if os.path.exists(log):
        with open(log) as f:
            assert b.check_tc_registers(f.read(), n) == 4  # D in {64, 128} x {bf16, f16}


SPILL_LOG = """ptxas info    : Compiling entry function '_ZN3foo16attn_simt_kernelIfLi128ELi8EEEv' for 'sm_103a'
ptxas info    : Function properties for _ZN3foo16attn_simt_kernelIfLi128ELi8EEEv
    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads
ptxas info    : Used 252 registers, used 1 barriers
ptxas info    : Compiling entry function '_ZN3foo12other_kernelEv' for 'sm_103a'
ptxas info    : Function properties for _ZN3foo12other_kernelEv
    8 bytes stack frame, 8 bytes spill stores, 8 bytes spill loads
ptxas info    : Compiling entry function '_ZN3foo16attn_simt_kernelIfLi64ELi4EEEv' for 'sm_103a'
ptxas info    : Function properties for _ZN3foo16attn_simt_kernelIfLi64ELi4EEEv
    16 bytes stack frame, 12 bytes spill stores, 20 bytes spill loads
ptxas info    : Used 255 registers, used 1 barriers
"""


def test_spill_report_is_read_per_instantiation():
    got = b.spills(SPILL_LOG, "attn_simt_kernel")
    assert got == [("_ZN3foo16attn_simt_kernelIfLi128ELi8EEEv", 0, 0), ("_ZN3foo16attn_simt_kernelIfLi64ELi4EEEv", 12, 20)]


def test_cuda_core_kernel_does_not_spill():
    # The library built in this tree: every instantiation (fp32/bf16/f16 x D 64/128 x 4/8 rows per thread)
    # fits its registers.
    log = os.path.join(b.OUT_DIR, "attn_simt.cu.ptxas.txt")
    if not os.path.exists(log):
        pytest.skip("no ptxas report of the CUDA-core kernel in this tree")
    with open(log) as f:
        got = b.spills(f.read(), "attn_simt_kernel")
    assert len(got) == 12
    assert all(st == 0 and ld == 0 for _, st, ld in got), got


def test_non_positive_scale_is_refused_for_16_bit_inputs():
    from paged_kv_cache_181_gb300 import _lib as lib

    def call(dt, scale, flags):
        # Valid sizes and NULL pointers: the host checks decide before any pointer is used.
        return lib.lib.paged_attn_varlen(None, 4, 4, None, None, 1, 16, 2, 64, dt, None, 1, 1, None, None, 4, 16,
                                         scale, None, None, None, None, 0, flags, None)

    for dt in (lib.PKV_BF16, lib.PKV_F16):
        for scale in (0.0, -0.125):
            assert call(dt, scale, 0) == lib.PKV_ERR_UNSUPPORTED
            assert "PKV_FORCE_SIMT" in lib.last_error()
            assert lib.last_launches() == 0
            # Asked for by name, the CUDA-core kernel takes it: the call gets past the scale to the pointers.
            assert call(dt, scale, lib.PKV_FORCE_SIMT) == lib.PKV_ERR_INVALID_ARG
            assert "NULL" in lib.last_error()
    assert call(lib.PKV_F32, -0.125, 0) == lib.PKV_ERR_INVALID_ARG  # fp32 takes any finite scale
    assert call(lib.PKV_BF16, 0.125, 0) == lib.PKV_ERR_INVALID_ARG
