"""bench.py's link between ncu summaries and the kernel source: the traffic
lines under profiles/ are keyed by a hash of the kernel's code with comments
and whitespace aside, so a comment edit keeps them and a code edit drops them."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_code_text_drops_comments_and_keeps_strings():
    src = 'int a = 1;   // note\n/* block\n comment */ const char* s = "a//b /*x*/";\nchar q = \'/\';'
    assert bench.code_text(src) == 'int a = 1; const char* s = "a//b /*x*/"; char q = \'/\';'
    # whitespace and comments only: same text
    assert bench.code_text("x  =\n\t1; // one") == bench.code_text("x = 1;")
    # a code change: different text
    assert bench.code_text("x = 1;") != bench.code_text("x = 2;")
    # escaped quotes inside a string do not end it
    assert bench.code_text('s = "a\\"//b"; // c') == 's = "a\\"//b";'


def test_profiled_traffic_lines_match_the_current_code():
    sha = bench.source_sha("decode.cu", "pd_device.cuh")
    # the headline decode's DRAM bytes were captured on the code as it stands
    t = bench.profiled_traffic("paged_decode", sha)
    assert t is not None and 3.0e8 < t < 3.5e8
    for S in (8, 16, 32, 64):
        assert bench.profiled_traffic(f"paged_decode_shared_cow_S{S}", sha) is not None
    assert bench.profiled_traffic("paged_decode", "0" * 16) is None
