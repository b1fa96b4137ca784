"""Every kernel has a byte-for-byte test (no GPU needed to check the registry).

The Megatron-LM determinism developer reference (section 4.3) keeps a manifest
of every file that launches GPU kernels, each entry naming its bit-exact
tests or an exemption, and a CPU-only test that fails when a kernel file is
added without an entry.  This is that gate for this library: each CUDA source
lists its kernels and the GPU tests that compare them with the oracle (or, for
the atomic baseline, that check it is order-dependent); the test below fails
when a file, a `__global__` kernel or a named test is missing.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "invariant_gradient_reduction_gb300", "csrc")
TESTS = os.path.join(ROOT, "tests")

# file -> (kernels, tests that run them) or (None, reason) for files without kernels
MANIFEST = {
    "api.cu": (None, "host helpers only (status strings, launch counter, device queries); test_abi.py"),
    "atomic.cu": (["atomic_scatter_kernel", "cast_bf16_kernel"],
                  ["test_atomic_baseline_close_to_oracle", "test_atomic_baseline_bf16_and_index_errors",
                   "test_atomic_negative_control_differs_across_replays"]),
    "gather.cu": (["gather_reduce_kernel", "finish_kernel"],
                  ["test_scatter_small_matches_oracle", "test_full_size_parity", "test_cluster_plan_hot_rows",
                   "test_segment_size_changes_no_bit", "test_index_add_matches_oracle"]),
    "gather_async.cu": (["gather_async_kernel"], ["test_gather_path_changes_no_bit"]),
    "gather_bulk.cu": (["gather_bulk_kernel", "gather_ring_kernel"],
                       ["test_gather_path_changes_no_bit", "test_index_add_bulk_ring_matches_oracle",
                        "test_ring_kernel_edge_cases"]),
    "hash.cu": (["hash_kernel"], ["test_hash_matches_oracle"]),
    "noalloc.cu": (None, "launches the gather and finish kernels of gather.cu; "
                         "test_noalloc_matches_workspace_entry_point_twice"),
    "plan.cu": (["tile_count_kernel", "tile_offset_kernel", "radix_scatter_kernel", "dup_key_kernel",
                 "row_bounds_kernel", "units_count_kernel", "units_scan_kernel", "units_write_kernel"],
                ["test_plan_lists_match_oracle", "test_plan_errors", "test_physical_row_permutation_with_src_id"]),
    "plan_cluster.cu": (["plan_cluster_kernel", "plan_cluster_one_kernel"],
                        ["test_plan_lists_match_oracle", "test_plan_paths_give_same_bytes"]),
    "plan_radix.cu": (["rx_count_kernel", "rx_offset_kernel", "rx_scatter_kernel", "rx_units_count_kernel",
                       "rx_units_write_kernel"],
                      ["test_plan_lists_match_oracle", "test_plan_paths_give_same_bytes", "test_plan_errors",
                       "test_cluster_plan_hot_rows", "test_plan_zipf_hot_rows_and_work_list"]),
    "plan_owner.cu": (["plan_owner_kernel"],
                      ["test_plan_lists_match_oracle", "test_plan_paths_give_same_bytes", "test_plan_errors",
                       "test_cluster_plan_hot_rows"]),
    "route.cu": (["router_topk_kernel", "route_cluster_kernel", "route_rows_kernel", "route_combine_kernel"],
                 ["test_router_topk_matches_oracle", "test_router_topk_ties_and_special_values",
                  "test_route_plan_matches_oracle", "test_route_combine_matches_oracle"]),
    "splitk.cu": (["splitk_kernel", "splitk_two_chunk_kernel"], ["test_splitk_matches_oracle", "test_splitk_split_counts"]),
    "splitk_gemm.cu": (["splitk_gemm_kernel"], ["test_splitk_gemm_partials_exact_on_integers",
                                                "test_splitk_gemm_fold_matches_oracle"]),
}


def _kernels_in(path):
    """Names of the `__global__` functions of a source: the first identifier after each
    `__global__` that is followed by its parameter list (launch bounds and register caps may
    nest parentheses)."""
    text = re.sub(r"//[^\n]*|/\*.*?\*/", " ", open(path).read(), flags=re.S)  # comments out
    names = set()
    for m in re.finditer(r"__global__\s+void\b", text):
        rest = text[m.end():]
        while rest.lstrip().startswith(("__launch_bounds__", "__maxnreg__")):
            i = rest.index("(")
            depth = 0
            for j in range(i, len(rest)):
                depth += {"(": 1, ")": -1}.get(rest[j], 0)
                if depth == 0:
                    rest = rest[j + 1:]
                    break
        names.add(re.match(r"\s*(\w+)\s*\(", rest).group(1))
    return names


def _test_names():
    names = set()
    for fn in os.listdir(TESTS):
        if fn.startswith("test_") and fn.endswith(".py"):
            names |= set(re.findall(r"^def (test_\w+)\(", open(os.path.join(TESTS, fn)).read(), flags=re.M))
    return names


def test_every_cuda_file_is_registered():
    files = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    assert files, "no CUDA sources found"
    missing = [f for f in files if f not in MANIFEST]
    assert not missing, f"CUDA sources without a manifest entry: {missing}"
    stale = [f for f in MANIFEST if f not in files]
    assert not stale, f"manifest entries without a source: {stale}"


def test_every_kernel_is_listed_and_every_test_exists():
    tests = _test_names()
    for fn, (kernels, entry) in MANIFEST.items():
        found = _kernels_in(os.path.join(CSRC, fn))
        if kernels is None:
            assert not found, f"{fn} defines kernels {sorted(found)} but is registered without any"
            assert isinstance(entry, str) and entry
            continue
        assert found == set(kernels), f"{fn}: kernels {sorted(found)} vs manifest {sorted(kernels)}"
        absent = [t for t in entry if t not in tests]
        assert entry and not absent, f"{fn}: tests not found: {absent}"
