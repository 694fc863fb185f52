"""The bench's pass rules on CPU: which timed passes count as stalled, and which pass of several
is reported (single rank)."""
import bench


def test_a_pass_with_one_step_above_twice_its_median_is_stalled():
    assert not bench.stalled([1.0, 1.1, 1.05, 1.02], 1)
    assert bench.stalled([1.0, 1.1, 1.05, 5.0], 1)


def test_a_pass_slow_from_end_to_end_is_stalled_against_a_reference():
    ref = 1.08  # the graph-replayed pass's median step, ms
    assert not bench.stalled([1.1, 1.12, 1.09], 1, ref)
    assert bench.stalled([40.0, 41.0, 39.0], 1, ref)  # no single outlier, every step slow
    # a short step's host-synchronised end-to-end pass is judged against the floor, not the step
    assert not bench.stalled([0.05, 0.05, 0.06], 1, max(0.03, bench.SLOW_FLOOR_MS))


def test_the_clean_pass_is_reported_else_the_lowest_median():
    assert bench.pick_pass([[5.0, 5.0], [1.0, 1.0]], True, 1) == 1  # the last, clean
    assert bench.pick_pass([[5.0, 5.0], [1.0, 9.0, 1.0], [3.0, 3.0]], False, 1) == 1


def test_kernel_code_hash_ignores_comments_and_whitespace(tmp_path):
    """A profile record stays valid across comment and layout edits of its kernel source, and
    no longer matches once the code itself changes."""
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("// a kernel\n__global__ void k(int* x) { x[0] = 1; }\n")
    b.write_text("__global__ void k(int* x) {\n  // set it\n  x[0] = 1;  // one\n}\n")
    c.write_text("__global__ void k(int* x) { x[0] = 2; }\n")
    assert bench.kernel_code_hash(str(a)) == bench.kernel_code_hash(str(b))
    assert bench.kernel_code_hash(str(a)) != bench.kernel_code_hash(str(c))
