"""Host-side bookkeeping of bench.py: the per-kernel code hashes that decide
whether the committed DRAM-traffic counters still describe the kernels."""

import os

import bench


def test_code_hash_ignores_comments_only():
    src = b"// header\n__global__ void k(int* p) {  /* block\n comment */\n  p[0] = 1;  // trailing\n}\n"
    same = b"__global__ void k(int* p) {\n\n  p[0] = 1;\n}\n// new comment\n"
    other = b"__global__ void k(int* p) {\n  p[0] = 2;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)


def test_phase_files_exist_for_both_head_dim_families():
    csrc = os.path.join(bench.ROOT, "bwd_flashattention_fwd_gb300", "csrc")
    for table in (bench.KERNEL_FILES, bench.KERNEL_FILES_D256):
        assert set(table) == {"fwd", "delta", "bwd_dkv", "bwd_dq"}
        for name in table.values():
            assert os.path.exists(os.path.join(csrc, name)), name
    # the D = 256 phases hash their own kernels, not the D <= 128 ones
    assert bench.kernel_source_hash("bwd_dkv", 256) != bench.kernel_source_hash("bwd_dkv", 128)
    assert bench.kernel_source_hash("delta", 256) == bench.kernel_source_hash("delta", 128)


def test_traffic_file_lines_are_well_formed():
    with open(bench.TRAFFIC_FILE) as f:
        lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert lines
    for kernel, workload, nbytes, h in lines:
        assert kernel in bench.KERNEL_FILES
        assert int(nbytes) > 0
        assert len(h) == 16 and int(h, 16) >= 0


def test_clock_window_keeps_samples_inside_the_region():
    c = bench.ClockSampler(0)
    c.proc = object()  # stands in for the running tool
    row = lambda mhz, cap: ["t", str(mhz), "2070", "500", "0x0", "Not Active", "Not Active", "Not Active", cap]
    c.samples = [(0.9, row(1000, "Not Active")), (1.02, row(2070, "Not Active")), (1.04, row(1900, "Active")),
                 (1.2, row(1500, "Not Active"))]
    c.t_begin, c.t_end = 1.0, 1.03
    wnd = c.window()
    assert wnd["samples"] == 2 and wnd["sm_mhz"] == (2070 + 1900) / 2
    assert wnd["reasons"] == ["sw_power_cap"]
    assert c.window(0.0, 0.95)["sm_mhz"] == 1000
