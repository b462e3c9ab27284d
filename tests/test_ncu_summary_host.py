"""The Nsight Compute summaries behind profiles/ (no GPU): launch lists with
mixed time units and tool chatter, and a raw counter page."""
from decode_megakernel_persistent_gb300 import ncu_summary

HDR = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
       '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n')


def row(i, kernel, unit, value, metric="gpu__time_duration.sum"):
    return (f'"{i}","1","python3","host","{kernel}","1","13","(544, 1, 1)","(152, 1, 1)","0","10.3",'
            f'"Command line profiler metrics","{metric}","{unit}","{value}"\n')


def test_launch_list_totals_and_shares(tmp_path):
    p = tmp_path / "launches.csv"
    p.write_text("==PROF== Connected to process 1\n" + HDR +
                 row(0, "decode_megakernel<0>(KParams)", "ns", "600000") +
                 row(1, "decode_megakernel<0>(KParams)", "us", "600") +
                 row(2, "decode_megakernel<0>(KParams)", "ns", "1,000", metric="dram__bytes_read.sum") +
                 row(3, "other_kernel(int)", "msecond", "0.3") +
                 "==PROF== Disconnected from process 1\n")
    out = ncu_summary.launches(str(p)).splitlines()
    assert out[2] == "| decode_megakernel<0> | 2 | 1200.0 | 600.0 | 80.0% |"
    assert out[3] == "| other_kernel | 1 | 300.0 | 300.0 | 20.0% |"


def test_raw_counters_in_fixed_order(tmp_path):
    p = tmp_path / "raw.csv"
    p.write_text('"Kernel Name","dram__bytes_read.sum","gpu__time_duration.sum","not_listed"\n'
                 '"","Gbyte","us",""\n'
                 '"decode_megakernel","2.5","672.2","7"\n')
    out = ncu_summary.raw(str(p)).splitlines()
    assert out[2:] == ["| gpu__time_duration.sum | 672.2 | us |", "| dram__bytes_read.sum | 2.5 | Gbyte |"]


def test_metrics_one_row_per_launch(tmp_path):
    p = tmp_path / "m.csv"
    p.write_text(HDR +
                 row(0, "k_gemm<0>(GemmArgs)", "us", "10.5") +
                 row(0, "k_gemm<0>(GemmArgs)", "%", "41.2", metric="sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active") +
                 row(1, "k_gemm<1>(GemmArgs)", "us", "7.25") +
                 row(1, "k_gemm<1>(GemmArgs)", "%", "38", metric="sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"))
    out = ncu_summary.metrics(str(p)).splitlines()
    assert out[0] == ("| launch | kernel | gpu__time_duration.sum | "
                      "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active |")
    assert out[2] == "| 0 | k_gemm<0> | 10.5 us | 41.2 % |"
    assert out[3] == "| 1 | k_gemm<1> | 7.25 us | 38 % |"
