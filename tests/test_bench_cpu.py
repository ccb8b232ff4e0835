"""Host-side pieces of bench.py: the source hash that keys the committed DRAM
traffic records ignores comment edits and notices code edits."""
import bench


def test_source_hash_ignores_comments_only():
    code = "int f(int a) {  // doubles\n    return 2 * a;\n}\n"
    recommented = "// header\nint f(int a) {  // twice a\n\n    return 2 * a;   \n}\n"
    edited = "int f(int a) {  // doubles\n    return 3 * a;\n}\n"
    assert bench.source_hash(code) == bench.source_hash(recommented)
    assert bench.source_hash(code) != bench.source_hash(edited)
    assert len(bench.source_hash(code)) == 16


def test_traffic_records_are_well_formed():
    # the records bench.py accepts for the current GEMM source (those whose
    # hash matches it) carry positive traffic above the weights' bytes
    recs = bench.traffic_record("gemm_tcgen05.cu")
    assert recs is not None
    for r in recs:
        assert r["dram_bytes_per_launch"] > r.get("weight_bytes", 0)
