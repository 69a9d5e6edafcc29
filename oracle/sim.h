/*
 * C interface of the C++ oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, single-threaded C++17 simulation of N ranks that run the
 * collective schedules of three source pages step by step, exchanging
 * messages:
 *   - the Bcast/Scatter page, "一对多通信：Broadcast 与 Scatter";
 *   - the hccl article (CSDN, CANN hccl's AllReduce algorithms), sections
 *     "Ring算法", "Mesh算法", "Tree算法";
 *   - the latency-formula page, "集合通信算法延迟公式".
 * Only the tests, the smoke check and the benchmark's CPU-baseline and
 * reference legs load it.  The CUDA library never includes, links or calls
 * it, and it includes nothing of the CUDA library.
 *
 * Element types (dtype): 0 fp32, 1 bf16, 2 int32, 3 fp16.  Ops: 0 sum,
 * 1 max, 2 min.  Buffers are the storage bytes of `count` elements.
 * Every call returns 0 on success, 1 when the schedule is not defined for the
 * arguments (an unknown algorithm for the collective), 2 for invalid
 * arguments; `err` (may be null) then holds a message.
 */
#ifndef VC_ORACLE_SIM_H_
#define VC_ORACLE_SIM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct vo_result vo_result;

/* One collective.  coll: "allreduce", "reduce_scatter", "allgather",
 * "broadcast", "scatter", "gather", "reduce", "alltoall".  inputs[r] holds
 * n_in elements per rank (broadcast and scatter: inputs[0] is the root's
 * buffer).  nranks is N.  nchunks is the pipelined broadcasts' chunk count
 * (algo "pipe_chain" / "pipe_tree"), ignored otherwise. */
int vo_run(const char* coll, const char* algo, int nranks, const void* const* inputs, int64_t n_in,
           int dtype, int op, int root, int inplace, int nchunks, vo_result** out, char* err, int errlen);

int vo_noutputs(const vo_result* r);
int64_t vo_output_elems(const vo_result* r, int i);
void vo_output_copy(const vo_result* r, int i, void* dst);
int64_t vo_hbm_bytes(const vo_result* r);
int vo_local_steps(const vo_result* r);
/* Transfer log: one record per message, 9 int64 fields each: step, src, dst,
 * n, reduce, esize, src_off (-1: none), dst_off (-1: none), chunk count. */
int64_t vo_nrecords(const vo_result* r);
void vo_records(const vo_result* r, int64_t* fields);
int64_t vo_nchunks_total(const vo_result* r);
void vo_record_chunks(const vo_result* r, int64_t* chunks);
const char* vo_record_phase(const vo_result* r, int64_t i);
void vo_free(vo_result* r);

/* Test-only fault injection: kind 1 loses every message of `step`, kind 2
 * delivers every message of `step` twice; kind 0 clears it. */
void vo_set_fault(int kind, int step);

/* Closed-form association trees, evaluated per element.  values[r] holds
 * rank r's stored input at the sampled element indices idx[0..nidx);
 * out receives the stored results.  AllReduce: algo fused, mesh, ring,
 * ring_hop, rhd, dbt, over buffers of `count` elements.  ReduceScatter:
 * algo fused or ring, element e of the N*rc input. */
int vo_allreduce_at(const void* const* values, int nranks, const char* algo, int64_t count, int dtype,
                    const int64_t* idx, int64_t nidx, int op, void* out, char* err, int errlen);
int vo_reduce_scatter_at(const void* const* values, int nranks, const char* algo, int64_t rc, int dtype,
                         const int64_t* idx, int64_t nidx, int op, void* out, char* err, int errlen);

/* The element conversions, exposed for pinning against library routines. */
void vo_bf16_from_f32(const float* x, uint16_t* out, int64_t n);
void vo_f32_from_bf16(const uint16_t* x, float* out, int64_t n);
void vo_f16_from_f32(const float* x, uint16_t* out, int64_t n);
void vo_f32_from_f16(const uint16_t* x, float* out, int64_t n);

#ifdef __cplusplus
}
#endif

#endif /* VC_ORACLE_SIM_H_ */
