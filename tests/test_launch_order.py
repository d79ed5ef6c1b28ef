"""Launch order of the CUDA kernels (source check, no GPU).

Kernels launched with programmatic dependent launch start before their predecessor has finished.
Every kernel of the library keeps one rule that makes a chain of such launches safe: it lets the
next kernel launch (griddep_launch_dependents) only after its own griddep_wait has returned, so a
kernel that starts early finds every kernel before its predecessor complete.  This test reads each
__global__ function of csrc/*.cu and checks that a griddep_wait precedes its first
griddep_launch_dependents.
"""

import pathlib
import re

CSRC = pathlib.Path(__file__).resolve().parents[1] / "bit_quantized_fine_nf4_b300" / "csrc"


def _global_bodies(text):
    """(name, body) of every __global__ function definition in `text` (brace matching)."""
    out = []
    for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\s*\([^)]*\)\s*)?(\w+)\s*\(", text):
        i = text.find("{", m.end())
        semi = text.find(";", m.end())
        if i < 0 or (0 <= semi < i and text[m.end():semi].count("(") <= text[m.end():semi].count(")")):
            continue  # a declaration
        depth, j = 0, i
        while j < len(text):
            if text[j] == "{":
                depth += 1
            elif text[j] == "}":
                depth -= 1
                if depth == 0:
                    break
            j += 1
        out.append((m.group(1), text[i:j + 1]))
    return out


def _strip_comments(text):
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def test_kernels_wait_before_letting_dependents_launch():
    checked = 0
    for f in sorted(CSRC.glob("*.cu")):
        for name, body in _global_bodies(_strip_comments(f.read_text())):
            trig = body.find("griddep_launch_dependents()")
            if trig < 0:
                continue
            wait = body.find("griddep_wait()")
            assert 0 <= wait < trig, f"{f.name}:{name} lets dependents launch before its griddep_wait"
            checked += 1
    assert checked >= 8, checked  # the kernels that trigger: side / grad / U / elementwise / decode / pair


def test_scanner_sees_a_violation():
    """The check itself: a kernel that triggers first is reported."""
    bad = """__global__ void k_bad(int* p) {
  griddep_launch_dependents();
  griddep_wait();
  *p = 1;
}
__global__ void k_good(int* p) {
  griddep_wait();
  griddep_launch_dependents();
}
"""
    bodies = dict(_global_bodies(bad))
    assert set(bodies) == {"k_bad", "k_good"}
    b = bodies["k_bad"]
    assert b.find("griddep_launch_dependents()") < b.find("griddep_wait()")
    g = bodies["k_good"]
    assert g.find("griddep_wait()") < g.find("griddep_launch_dependents()")
