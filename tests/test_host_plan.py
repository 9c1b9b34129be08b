"""The launch plan's host-side rules (csrc/gemm_plan.h, csrc/gemm_params.h), compiled for the
host and checked on the CPU: the stream-K partition helpers against the
scheduler model (oracle/sched.py, which writes the partition out k-block by
k-block), and the thresholds and shared-memory budget the launcher uses."""
import json
import os
import shutil
import subprocess
import tempfile

import pytest

from oracle import sched as sm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "persistent_tile_scheduled_gb300", "csrc")

CASES = [(5, 3, 4), (7, 3, 1), (104, 76, 64), (256, 76, 64), (300, 152, 5), (31, 16, 9), (1024, 76, 128),
         (28, 28, 3), (77, 76, 2)]

PROGRAM = r"""
#include <cstdio>
#include "gemm_plan.h"
using namespace pts;
int main() {
    const long long cases[][3] = {%CASES%};
    int first = 1;
    printf("{\"cases\": [");
    for (unsigned i = 0; i < sizeof(cases) / sizeof(cases[0]); ++i) {
        const long long T = cases[i][0], G = cases[i][1], kb = cases[i][2];
        const long long sk1 = choose_stream_k(T, G, kb, 1), sk0 = choose_stream_k(T, G, kb, 0),
                        skn = choose_stream_k(T, G, kb, -1);
        printf("%s{\"T\": %lld, \"G\": %lld, \"kb\": %lld, \"sk_force\": %lld, \"sk_auto\": %lld, \"sk_never\": %lld",
               i ? ", " : "", T, G, kb, sk1, sk0, skn);
        const long long L = sk1 * kb;
        printf(", \"begin\": [");
        for (long long c = 0; sk1 && c < G; ++c) printf("%s%lld", c ? ", " : "", (long long)sk_unit_begin(c, L, G));
        printf("], \"pieces\": [");
        for (long long c = 0; sk1 && c < G; ++c) printf("%s%d", c ? ", " : "", sk_pieces(c, L, G, kb));
        printf("], \"owner\": [");
        for (long long x = 0; x < L; ++x) printf("%s%lld", x ? ", " : "", (long long)sk_unit_of(x, L, G));
        printf("]}");
    }
    printf("], \"split\": [");
    const long long sp[][2] = {{8, 152}, {38, 152}, {39, 152}, {76, 152}, {77, 152}, {151, 152}, {152, 152}, {500, 152}};
    for (unsigned i = 0; i < sizeof(sp) / sizeof(sp[0]); ++i)
        printf("%s[%lld, %lld, %d]", i ? ", " : "", sp[i][0], sp[i][1], choose_split(sp[i][0], sp[i][1]));
    printf("], \"cta_group\": [");
    for (int kb = 1; kb <= 40; ++kb) printf("%s%d", kb > 1 ? ", " : "", choose_cta_group(kb));
    printf("], \"cta_group_np\": [");
    for (int kb = 1; kb <= 80; ++kb) printf("%s%d", kb > 1 ? ", " : "", choose_cta_group(kb, SCHED_NONPERSISTENT));
    printf("], \"cta_group_clc\": [");
    for (int kb = 1; kb <= 40; ++kb) printf("%s%d", kb > 1 ? ", " : "", choose_cta_group(kb, SCHED_CLC));
    printf("], \"last_wave\": [");
    const long long lw[][2] = {{256, 76}, {512, 152}, {1024, 76}, {270, 76}, {304, 76}, {300, 76}, {76, 76},
                               {40, 76}, {5, 3}, {7, 3}, {114, 76}, {115, 76}, {400, 76}};
    first = 1;
    for (unsigned i = 0; i < sizeof(lw) / sizeof(lw[0]); ++i)
        for (int kb = 2; kb <= 130; kb += 4)
            for (int aut = 0; aut <= 1; ++aut)
                for (int f = -1; f <= 1; ++f)
                    for (int sched = 0; sched <= 2; ++sched) {
                        int64_t tail = -7;
                        const long long sk = choose_last_wave(lw[i][0], lw[i][1], kb, aut != 0, f, sched, tail);
                        printf("%s[%lld, %lld, %d, %d, %d, %d, %lld, %lld]", first ? "" : ", ", lw[i][0], lw[i][1], kb,
                               aut, f, sched, sk, (long long)tail);
                        first = 0;
                    }
    printf("], \"tail_max_kb\": %d", kTailMaxKb);
    printf(", \"pair_min_kb\": %d, \"pair_min_kb_np\": %d, \"sk_min_saved_kb\": %d", kPairMinKb,
           kPairMinKbNonPersistent, kSkMinSavedKb);
    printf(", \"kb_per_stage\": [%d, %d], \"smem\": [%d, %d, %d]", kb_per_stage(1), kb_per_stage(2),
           smem_bytes(1, 4), smem_bytes(2, 3), smem_bytes(1, 5));
    printf(", \"narrow\": {\"smem\": %d, \"smem3\": %d, \"stages\": %d, \"per_sm\": [%d, %d, %d, %d], "
           "\"pair_smem\": [%d, %d], \"max_kb\": %d, \"tile\": [",
           smem_bytes(1, kNarrowStages, kTileNNarrow), smem_bytes(1, 3, kTileNNarrow), kNarrowStages,
           ctas_per_sm(1, kTileN), ctas_per_sm(2, kTileN), ctas_per_sm(1, kTileNNarrow), ctas_per_sm(2, kTileNNarrow),
           smem_bytes(2, 4, kTileNNarrow), smem_bytes(2, 5, kTileNNarrow), kNarrowMaxKb);
    first = 1;
    for (int kb = 1; kb <= 10; ++kb)
        for (int cg = 0; cg <= 2; ++cg)
            for (int sched = 0; sched <= 2; ++sched) {
                printf("%s[%d, %d, %d, %d]", first ? "" : ", ", kb, cg, sched, choose_tile_n(kb, cg, sched));
                first = 0;
            }
    printf("]}}\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def plan():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc is needed to compile the host program")
    src = PROGRAM.replace("%CASES%", ", ".join("{%d, %d, %d}" % c for c in CASES))
    with tempfile.TemporaryDirectory() as d:
        cu, exe = os.path.join(d, "plan.cu"), os.path.join(d, "plan")
        open(cu, "w").write(src)
        subprocess.run([nvcc, "-std=c++17", "-I", CSRC, cu, "-o", exe], check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return json.loads(out)


def test_stream_k_partition_matches_the_model(plan):
    for case in plan["cases"]:
        T, G, kb, sk = case["T"], case["G"], case["kb"], case["sk_force"]
        R = T % G
        assert sk == (R + G if T >= G and R else 0), case
        assert case["sk_never"] == 0
        if not sk:
            continue
        units = sm.work_units(T, num_kb=kb, sk_tiles=sk, sk_units=G)
        L = sk * kb
        for c in range(G):
            items = units[c]
            assert case["pieces"][c] == len(items), (case, c)
            # the unit's first k-block of the region: its last-run piece is its first tile
            t, k0 = items[-1][1], items[-1][4]
            assert case["begin"][c] == t * kb + k0, (case, c)
        owner = [None] * L
        for c in range(G):
            for _, t, _, _, k0, k1 in units[c]:
                for k in range(k0, k1):
                    owner[t * kb + k] = c
        assert case["owner"] == owner, case


def test_stream_k_is_used_only_when_it_saves_enough(plan):
    m = plan["sk_min_saved_kb"]
    for case in plan["cases"]:
        T, G, kb = case["T"], case["G"], case["kb"]
        R = T % G
        want = case["sk_force"] if (case["sk_force"] and kb * (G - R) >= m * G) else 0
        assert case["sk_auto"] == want, case


def test_last_wave_halves_or_stream_k(plan):
    """The partial last wave of T tiles on G clusters (R = T mod G): its R tiles
    run as column halves under the persistent schedulers when 2R <= G and
    the caller left slicing to the library, unless the stream-K share is
    forced or the tiles are long enough (tail_max_kb k-blocks) for the share,
    where it saves enough, to be used instead; never both."""
    m, tmax = plan["sk_min_saved_kb"], plan["tail_max_kb"]
    seen = set()
    for T, G, kb, aut, force, sched, sk, tail in plan["last_wave"]:
        R = T % G
        halves = R if (aut and sched != 0 and T > G and R and 2 * R <= G) else 0
        share = R + G if (T >= G and R) else 0
        if force < 0:
            want_sk = 0
        elif force > 0:
            want_sk = share
        else:
            want_sk = share if (share and kb * (G - R) >= m * G and not (halves and kb < tmax)) else 0
        assert sk == want_sk, (T, G, kb, aut, force, sched)
        assert tail == (0 if want_sk else halves), (T, G, kb, aut, force, sched)
        seen.add((bool(sk), bool(tail)))
    assert seen == {(False, False), (True, False), (False, True)}


def test_slices_and_cta_group_thresholds(plan):
    for tiles, resident, split in plan["split"]:
        want = 1 if tiles >= resident else (4 if 4 * tiles <= resident else (2 if 2 * tiles <= resident else 1))
        assert split == want, (tiles, resident)
    k = plan["pair_min_kb"]
    assert plan["cta_group"] == [2 if kb >= k else 1 for kb in range(1, 41)]
    assert plan["cta_group_clc"] == plan["cta_group"]
    # the non-persistent grid keeps single CTAs much longer (a pair cluster per tile costs more)
    knp = plan["pair_min_kb_np"]
    assert knp > k
    assert plan["cta_group_np"] == [2 if kb >= knp else 1 for kb in range(1, 81)]


def test_shared_memory_budget(plan):
    single, pair, five = plan["smem"]
    assert plan["kb_per_stage"] == [1, 2]
    # the default rings (4 single-CTA stages, 3 pair stages) fit the 227 KB a CTA may use; a
    # fifth single-CTA stage does not
    assert single <= 232448 and pair <= 232448 and five > 232448


def test_narrow_tile_rules(plan):
    """The narrow tile's ring, staging and barriers fit twice in an SM's 228 KB
    with the 1 KB each CTA reserves (a third stage would not); its pair form
    runs one CTA per SM, with a ring of four two-k-block stages (48 KB each:
    128 rows of A and 64 of B per k-block) in the 227 KB a CTA may use (a fifth
    would not fit); the library picks the narrow tile only for the
    non-persistent grid, on tiles of at most 4 k-blocks, when the CTA group is
    left to it (so never the pair form)."""
    n = plan["narrow"]
    assert n["stages"] == 2 and n["per_sm"] == [1, 1, 2, 1]
    assert 2 * (n["smem"] + 1024) <= 233472 < 2 * (n["smem3"] + 1024)
    four, five = n["pair_smem"]
    assert four <= 232448 < five
    assert five - four == 2 * (128 + 64) * 128
    assert n["max_kb"] == 4
    for kb, cg, sched, tile in n["tile"]:
        want = 128 if (cg == 0 and sched == 0 and kb <= 4) else 256
        assert tile == want, (kb, cg, sched)
