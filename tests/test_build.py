"""The build's register guard (CPU only). The forward kernel splits its registers
between warpgroups with setmaxnreg, assuming 168 registers per thread at
launch (384 threads); a different allocation would leave a warpgroup waiting
for registers that never come, so the build must refuse it. Also checks that
the library actually built here passed that guard."""
import pytest

from exact_attention_91_gb300 import build as fb

GOOD = """
ptxas info    : Compiling entry function '_ZN2fa13fa_fwd_kernelILi128ELb1ELb0EEEv14CUtensorMap_stS1_S1_S1_NS_9FwdParamsE' for 'sm_103a'
ptxas info    : Function properties for _ZN2fa13fa_fwd_kernelILi128ELb1ELb0EEEv14CUtensorMap_stS1_S1_S1_NS_9FwdParamsE
    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads
ptxas info    : Used 168 registers, used 16 barriers
ptxas info    : Compiling entry function '_ZN2fa13fa_fwd_kernelILi64ELb0ELb1EEEv14CUtensorMap_stS1_S1_S1_NS_9FwdParamsE' for 'sm_103a'
    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads
ptxas info    : Used 168 registers, used 16 barriers
ptxas info    : Compiling entry function '_Z26fa_selftest_timeout_kernely' for 'sm_103a'
ptxas info    : Used 11 registers, used 0 barriers, 16 bytes smem
"""


def test_report_with_the_assumed_register_count_passes():
    regs = fb.check_ptxas_report(GOOD)
    assert sorted(regs.values()) == [11, 168, 168]


def test_a_different_register_count_is_refused():
    with pytest.raises(RuntimeError, match="168"):
        fb.check_ptxas_report(GOOD.replace("Used 168 registers", "Used 160 registers", 1))


def test_a_report_without_the_kernel_is_refused():
    only_selftest = GOOD.split("ptxas info    : Compiling entry function '_Z26")[1]
    with pytest.raises(RuntimeError, match="fa_fwd_kernel"):
        fb.check_ptxas_report("ptxas info    : Compiling entry function '_Z26" + only_selftest)


def test_every_split_kernel_is_guarded():
    assert set(fb.LAUNCH_REGS) == {"fa_fwd_kernel"}
    assert all(v == 168 for v in fb.LAUNCH_REGS.values())
