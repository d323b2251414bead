// ar_comm.cpp — a host-side communicator for virtual ranks that are host
// threads: each thread submits its rank's half of a collective; the call
// launches once every rank has arrived with the same arguments.
//
// "All-Reduce・All-Gather・All-to-Allとは？" (vasteelab), §rankとcommunicator:
// every rank must call the matching collective with the same count and data
// type or the collective may hang, crash or corrupt data; §hangをtimeoutだけで
// 再起動しない: hangs come from ranks that skip a call, differing counts or
// types, mismatched groups, an earlier error, or a different call order, and
// each rank's last collective, sequence number, shape, data type,
// communicator id and earlier error should be recorded. Here a mismatch is
// detected before anything is launched (AR_ERR_MISMATCH for every rank of
// that call), a rank that never arrives ends the wait of the others after
// the communicator's timeout (AR_ERR_TIMEOUT), and either error poisons the
// communicator: later calls return it at once, so a group is isolated
// instead of silently continuing. Waits are host waits only; no kernel waits
// on another rank.
#include <chrono>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <vector>

#include "ar.h"
#include "ar_internal.h"

namespace {

using clk = std::chrono::steady_clock;

struct Desc {
  int collective;
  size_t count;
  int dtype, op, algo;
  ar_stream_t stream;
  bool operator==(const Desc& o) const {
    return collective == o.collective && count == o.count && dtype == o.dtype && op == o.op && algo == o.algo &&
           stream == o.stream;
  }
};

struct Round {
  Desc desc{};
  int arrived = 0, left = 0;
  uint64_t arrived_mask = 0, mismatch_mask = 0;
  bool decided = false;
  ar_status_t status = AR_SUCCESS;
  clk::time_point first{}, last{};
  std::vector<const void*> send;
  std::vector<void*> recv;
};

}  // namespace

struct ar_comm {
  int nranks = 0;
  int timeout_ms = 0;
  uint64_t id = 0;
  bool log = false;
  std::mutex mu;
  std::condition_variable cv;
  std::vector<uint64_t> seq;               // per rank: collectives entered
  std::map<uint64_t, Round> rounds;        // by sequence number
  ar_status_t poisoned = AR_SUCCESS;
  std::vector<ar_call_record_t> records;   // per rank: the last collective
};

namespace {

uint64_t next_comm_id() {
  static std::mutex m;
  static uint64_t n = 0;
  std::lock_guard<std::mutex> g(m);
  return ++n;
}

void record(ar_comm* c, int rank, uint64_t seq, const Desc& d, ar_status_t st, const Round* R) {
  ar_call_record_t& rec = c->records[rank];
  rec.comm_id = c->id;
  rec.seq = seq;
  rec.collective = d.collective;
  rec.count = d.count;
  rec.dtype = d.dtype;
  rec.op = d.op;
  rec.algo = d.algo;
  rec.status = st;
  rec.arrived_mask = R ? R->arrived_mask : 0;
  rec.mismatch_mask = R ? R->mismatch_mask : 0;
  rec.arrival_skew_ms =
      (R && R->arrived > 0) ? std::chrono::duration<double, std::milli>(R->last - R->first).count() : 0.0;
  if (c->log)
    std::fprintf(stderr, "[ar comm %llu] rank %d seq %llu allreduce count %zu dtype %d op %d algo %d -> %s\n",
                 (unsigned long long)c->id, rank, (unsigned long long)seq, d.count, d.dtype, d.op, d.algo,
                 ar_status_string(st));
}

}  // namespace

extern "C" {

ar_status_t ar_comm_create(int nranks, int timeout_ms, ar_comm_t** comm) {
  if (!comm || nranks < 1 || nranks > AR_MAX_RANKS || timeout_ms < 0) return AR_ERR_INVALID_ARGUMENT;
  ar_comm* c = new ar_comm();
  c->nranks = nranks;
  c->timeout_ms = timeout_ms;
  c->id = next_comm_id();
  const char* dbg = std::getenv("AR_DEBUG");
  c->log = dbg && dbg[0] && dbg[0] != '0';
  c->seq.assign(nranks, 0);
  c->records.assign(nranks, ar_call_record_t{});
  *comm = c;
  return AR_SUCCESS;
}

ar_status_t ar_comm_destroy(ar_comm_t* comm) {
  if (!comm) return AR_ERR_INVALID_ARGUMENT;
  delete comm;
  return AR_SUCCESS;
}

ar_status_t ar_comm_allreduce(ar_comm_t* c, int rank, const void* sendbuf, void* recvbuf, size_t count,
                              ar_dtype_t dtype, ar_op_t op, ar_algo_t algo, ar_stream_t stream) {
  if (!c || rank < 0 || rank >= c->nranks) return AR_ERR_INVALID_ARGUMENT;
  const Desc d{1, count, (int)dtype, (int)op, (int)algo, stream};
  std::unique_lock<std::mutex> lk(c->mu);
  const uint64_t seq = ++c->seq[rank];
  if (c->poisoned != AR_SUCCESS) {
    record(c, rank, seq, d, c->poisoned, nullptr);
    return c->poisoned;
  }
  Round& R = c->rounds[seq];
  const clk::time_point now = clk::now();
  if (R.arrived == 0 && !R.decided) {
    R.desc = d;
    R.first = now;
    R.send.assign(c->nranks, nullptr);
    R.recv.assign(c->nranks, nullptr);
  }
  R.last = now;
  ar_status_t st;
  if (R.decided) {  // the call already failed (a late arrival)
    st = R.status;
  } else if (!(d == R.desc)) {
    R.mismatch_mask |= 1ull << rank;
    R.arrived_mask |= 1ull << rank;
    R.arrived += 1;
    R.decided = true;
    R.status = st = AR_ERR_MISMATCH;
    c->poisoned = st;
    c->cv.notify_all();
  } else {
    R.send[rank] = sendbuf;
    R.recv[rank] = recvbuf;
    R.arrived_mask |= 1ull << rank;
    R.arrived += 1;
    if (R.arrived == c->nranks) {  // the last arrival launches the one device call
      st = ar_allreduce(R.send.data(), R.recv.data(), c->nranks, count, dtype, op, algo, stream);
      R.decided = true;
      R.status = st;
      if (st != AR_SUCCESS) c->poisoned = st;
      c->cv.notify_all();
    } else {
      const clk::time_point deadline = now + std::chrono::milliseconds(c->timeout_ms);
      if (!c->cv.wait_until(lk, deadline, [&] { return R.decided; })) {
        R.decided = true;
        R.status = AR_ERR_TIMEOUT;
        c->poisoned = AR_ERR_TIMEOUT;
        c->cv.notify_all();
      }
      st = R.status;
    }
  }
  record(c, rank, seq, d, st, &R);
  R.left += 1;
  if (R.left == c->nranks) c->rounds.erase(seq);  // every rank has seen the outcome
  return st;
}

ar_status_t ar_comm_last_record(ar_comm_t* c, int rank, ar_call_record_t* out) {
  if (!c || !out || rank < 0 || rank >= c->nranks) return AR_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> g(c->mu);
  *out = c->records[rank];
  return AR_SUCCESS;
}

}  // extern "C"
